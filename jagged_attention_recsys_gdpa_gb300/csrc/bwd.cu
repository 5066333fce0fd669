// Backward pass of jagged generalized dot-product attention on sm_103a.
//
// "GEM Training" post, section "Jagged Sequence Flash Attention", bullet on
// backward parallelisation: for many sequences x heads the fastest scheme is
// not to split a sequence's key range across CTAs and to compute dQ in its
// own pass (split dQ / dK-dV), so that no atomic adds are needed. Here:
//   dq    one item = (sequence, 128-query tile, head); walks its key tiles:
//         S = Q K^T, dP = dO V^T, dS, dQ += dS K. For softmax its warps 2-3
//         also compute Di = rowsum(dO * O) per query row and head (section
//         "BlockAttention" of the same post names the separate Di
//         preprocessing pass of FlashAttention, which this removes), so it
//         runs first and the dK/dV pass reads Di.
//   dkdv  one item = (sequence, 128-key tile, head); walks the query tiles
//         that can see it: S^T = K Q^T, dP^T = V dO^T, P^T and dS^T from the
//         activation, dV += P^T dO, dK += dS^T Q (all accumulated in TMEM)
// Both MMA kernels are persistent and warp-specialised: warp 0 issues TMA
// copies, warp 1 issues tcgen05 MMAs, and two activation warpgroups (warps
// 4-7 and 8-11; one TMEM lane per thread) split every 128-column score tile
// in halves, apply the activation and its derivative, and write P / dS back
// to TMEM as bf16 in their own column ranges, where the next MMA reads them
// as its A operand. Two warps per scheduler hide the latency of the
// transcendental and conversion instructions that one warp cannot. An
// epilogue warpgroup (warps 12-15) drains each item's accumulators (dQ, or
// dV then dK, each released to the MMAs as soon as it is read) while the
// activation warpgroups already work on the next item.
#include <cstdint>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

// Compiled twice: on its own, and through bwd_hilo.cu with JATTN_HILO = 1 for
// pointwise activations without the 1/Lkv normaliser, whose P and dS enter the
// second products as bf16 hi + lo parts (kept out of the other kernels, where
// even untaken branches for them cost code quality in the activation loops).
#ifndef JATTN_HILO
#define JATTN_HILO 0
#endif

namespace jattn {

namespace {

// warp 0 TMA, warp 1 MMA, warps 2-3 Di (dQ) or LSE / Di staging (dK/dV;
// softmax), warps 4-11 activation, warps 12-15 epilogue
constexpr int kThreads = 512;
// Register split (setmaxnreg, per warpgroup): 512 x 128 at launch = 65536 =
// 128 x control + 256 x activation + 128 x epilogue, shares that compile
// without spills: the hi + lo kernels' MMA issuer needs more, their
// activation less.
#if JATTN_HILO
constexpr int kCtlRegs = 104;
constexpr int kActRegs = 168;
#else
constexpr int kCtlRegs = 88;
constexpr int kActRegs = 176;
#endif
constexpr int kEpiRegs = 72;
static_assert(128 * kCtlRegs + 256 * kActRegs + 128 * kEpiRegs <= 65536, "register split");
constexpr int kNG = 2;          // activation warpgroups; they split each score tile's columns
constexpr int kCols = kTile / kNG;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// act(x) and act'(x) for the pointwise activations.
template <int ACT>
__device__ __forceinline__ void act_and_grad(float x, float& f, float& g) {
  if constexpr (ACT == JATTN_SILU) {
    const float sg = __fdividef(1.0f, 1.0f + ex2_approx(-x * kLog2e));
    f = x * sg;
    g = sg * fmaf(x, 1.0f - sg, 1.0f);
  } else if constexpr (ACT == JATTN_GELU_POLY) {
    f = gelu_poly(x);
    g = gelu_poly_grad(x);
  } else {
    const float k0 = 0.7978845608028654f, k1 = 0.044715f;
    const float x2 = x * x;
    const float t = tanh_approx(k0 * fmaf(k1 * x2, x, x));
    f = 0.5f * x * (1.0f + t);
    g = fmaf(0.5f * x * (1.0f - t * t) * k0, fmaf(3.0f * k1, x2, 1.0f), 0.5f * (1.0f + t));
  }
}

// Store one 128-bit-vectorised bf16 row chunk of 32 fp32 values times `mul`.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&v)[32], float mul, int v8) {
  uint32_t w[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
  store_words16(dst, w, v8);
}

__device__ __forceinline__ void zero_row(__nv_bfloat16* dst, int D) {
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (int e = 0; e < D / 8; ++e) d[e] = make_uint4(0, 0, 0, 0);
}

// All 128 threads of an activation warpgroup meet on an mbarrier (count 128);
// the wait is bounded, so a warpgroup whose other warps have aborted gives up
// instead of hanging.
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& phase, volatile int* abort_flag,
                                           const AttnArgs& a, int where) {
  mbar_arrive(bar);
  const bool ok = wait_bar(bar, phase & 1, abort_flag, a, where);
  ++phase;
  return __all_sync(0xffffffffu, ok);
}

// Epilogue warpgroup: each thread stores its accumulator row, D/32 chunks of
// 32 columns read, rotated back (rc != nullptr), scaled and written with
// 32-byte stores; `release` is arrived once every column is read. (Staging
// whole tiles through shared memory for TMA stores, as the activation warps
// once did, made this warpgroup slow enough to stall the next item's MMAs.)
template <int D>
__device__ __forceinline__ void epi_rows(uint32_t tacc, float mul, __nv_bfloat16* dst, bool valid, uint64_t* release,
                                         const AttnArgs& a, const float* rc, const float* rs) {
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t v[32];
    tmem_ld32(tacc + c * 32, v);
    tmem_ld_wait();
    if (c == D / 32 - 1) {
      tc_fence_before();
      mbar_arrive(release);
    }
    if (rc != nullptr)
      rope_back16(v, rc + static_cast<int64_t>(16 * c) * a.rope_rows, rs + static_cast<int64_t>(16 * c) * a.rope_rows,
                  a.rope_rows);
    if (valid) store_row32(dst + c * 32, v, mul, a.out_v8);
  }
}

struct BwdItem {
  int b, rt, lo, hi, h, lq, lkv;
  int64_t q0, k0;
};

__device__ __forceinline__ bool load_bwd_item(const AttnArgs& a, long long round, BwdItem& it) {
  const long long n_items = static_cast<long long>(*a.n_tiles) * a.H;
  const long long k = zigzag_item(round, blockIdx.x, gridDim.x);
  if (k >= n_items) return false;
  const int4 t = a.tiles[k / a.H];
  it.h = static_cast<int>(k % a.H);
  it.b = t.x;
  it.rt = t.y;
  it.lo = t.z;
  it.hi = t.w;
  it.q0 = a.q_off[it.b];
  it.k0 = a.kv_off[it.b];
  it.lq = static_cast<int>(a.q_off[it.b + 1] - it.q0);
  it.lkv = static_cast<int>(a.kv_off[it.b + 1] - it.k0);
  return true;
}

// ---------------------------------------------------------------------------- dK / dV
// TMEM address of the A operand for K-step kk of a 128-column score tile
// whose bf16 pairs were written by the two activation warpgroups: group g
// packs score columns [64g, 64g+64) into TMEM columns [base+64g, base+64g+32).
__device__ __forceinline__ uint32_t split_a(uint32_t base, int kk) { return base + (kk >> 2) * 64 + (kk & 3) * 8; }

template <int D>
struct DkdvCfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = (D == 128) ? 2 : 3;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;                               // stage s: Q, then dO
  static constexpr int kLseOff = 2 * kTileBytes + kStages * 2 * kTileBytes;  // [2][128] lse2, [2][128] Di
  static constexpr int kBarOff = kLseOff + 4 * kTile * 4;
  static constexpr int kSmemBytes = kBarOff + 256;  // base 1024-aligned (checked)
  static constexpr uint32_t kSCol = 0, kDPCol = 128, kDVCol = 256, kDKCol = 256 + D;
};

struct DkdvBars {
  uint64_t kv_full, kv_empty;
  uint64_t qd_full[3], qd_empty[3];
  uint64_t s_full, dp_full, p_ready, ds_ready;
  uint64_t dv_full, dk_full, dv_empty, dk_empty;  // accumulators handed to / back from the epilogue warpgroup
  uint64_t drain;
  uint64_t ld_full[2], ld_empty[2];  // per-step LSE / Di slots (softmax), filled by warps 2-3
  uint32_t tmem_base;
  int abort_flag;
};

static_assert(sizeof(DkdvBars) <= 256, "barrier block overflows its slot");
static_assert(DkdvCfg<128>::kSmemBytes <= 227 * 1024 && DkdvCfg<64>::kSmemBytes <= 227 * 1024, "shared memory");

template <int D, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const AttnArgs a) {
  using C = DkdvCfg<D>;
  constexpr bool kHilo = JATTN_HILO && ACT != JATTN_SOFTMAX;  // P and dS as bf16 hi + lo parts
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned tiles and no slack for realigning: a misaligned base is an error
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(a.status, JATTN_ERR_UNSUPPORTED, 19, blockIdx.x);
    return;
  }
  uint8_t* sm = smem_raw;
  DkdvBars* bars = reinterpret_cast<DkdvBars*>(sm + C::kBarOff);
  float* s_lse = reinterpret_cast<float*>(sm + C::kLseOff);  // [2][128]
  float* s_di = s_lse + 2 * kTile;                           // [2][128]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->qd_full[s], 1);
      mbar_init(&bars->qd_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, kNG * kTile);
    mbar_init(&bars->ds_ready, kNG * kTile);
    mbar_init(&bars->dv_full, 1);
    mbar_init(&bars->dk_full, 1);
    mbar_init(&bars->dv_empty, kTile);  // the epilogue warpgroup's threads
    mbar_init(&bars->dk_empty, kTile);
    mbar_init(&bars->drain, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->ld_full[x], 64);
      mbar_init(&bars->ld_empty[x], kNG * kTile);
    }
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
    if (lane == 0) {
      uint32_t item_cnt = 0, qd_it = 0;
      bool kv_armed = false, ok = true;
      BwdItem it, nit;
      bool have = load_bwd_item(a, 0, it), have_next = false;
      for (long long r = 0; have && ok; ++r, it = nit, have = have_next) {
        have_next = load_bwd_item(a, r + 1, nit);  // in flight while this item is served
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->kv_empty, (item_cnt & 1) ^ 1, abort_flag, a, 40))) break;
        ++item_cnt;
        const int yk = static_cast<int>(it.k0) + it.rt * kTile;
        if (!(a.debug_flags & 1)) {
          mbar_arrive_expect_tx(&bars->kv_full, 2 * C::kTileBytes);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(sm + C::kKOff + c * kTile * 128, &tmK, &bars->kv_full, it.h * D + c * 64, yk);
            tma_load_2d(sm + C::kVOff + c * kTile * 128, &tmV, &bars->kv_full, it.h * D + c * 64, yk);
          }
          kv_armed = true;
        }
        for (int i = it.lo; i < it.hi; ++i, ++qd_it) {
          const int s = qd_it % C::kStages;
          if (!(ok = wait_bar(&bars->qd_empty[s], ((qd_it / C::kStages) & 1) ^ 1, abort_flag, a, 41))) break;
          const int yq = static_cast<int>(it.q0) + i * kTile;
          mbar_arrive_expect_tx(&bars->qd_full[s], 2 * C::kTileBytes);
          uint8_t* st = sm + C::kQOff + s * 2 * C::kTileBytes;
          for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(st + c * kTile * 128, &tmQ, &bars->qd_full[s], it.h * D + c * 64, yq);
            tma_load_2d(st + C::kTileBytes + c * kTile * 128, &tmDO, &bars->qd_full[s], it.h * D + c * 64, yq);
          }
        }
      }
      if (kv_armed) drain_wait(&bars->kv_full, (item_cnt - 1) & 1, a.timeout_ns);
      for (uint32_t i = (qd_it > (uint32_t)C::kStages ? qd_it - C::kStages : 0); i < qd_it; ++i)
        drain_wait(&bars->qd_full[i % C::kStages], (i / C::kStages) & 1, a.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kTile, kTile, false, false);
      constexpr uint32_t idAcc = idesc_bf16_f32(kTile, D, false, true);
      const uint32_t sK = smem_u32(sm + C::kKOff), sV = smem_u32(sm + C::kVOff);
      const uint32_t sQ0 = smem_u32(sm + C::kQOff);
      uint32_t item_cnt = 0, qd_it = 0, p_cnt = 0, ds_cnt = 0, acc_cnt = 0;
      bool ok = true;
      auto sQ = [&](int s) { return sQ0 + s * 2 * C::kTileBytes; };
      auto sDO = [&](int s) { return sQ0 + s * 2 * C::kTileBytes + C::kTileBytes; };
      auto kmajor = [](uint32_t base, int kk) {
        return sdesc_sw128(base + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16, 1024);
      };
      auto issue_s = [&](int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + C::kSCol, kmajor(sK, kk), kmajor(sQ(s), kk), idS, kk > 0);
        mma_commit(&bars->s_full);
      };
      auto issue_dp = [&](int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + C::kDPCol, kmajor(sV, kk), kmajor(sDO(s), kk), idS, kk > 0);
        mma_commit(&bars->dp_full);
      };
      BwdItem it, nit;
      bool have = load_bwd_item(a, 0, it), have_next = false;
      for (long long r = 0; have && ok; ++r, it = nit, have = have_next) {
        have_next = load_bwd_item(a, r + 1, nit);
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->kv_full, item_cnt & 1, abort_flag, a, 50))) break;
        ++item_cnt;
        tc_fence_after();
        {
          const int s = qd_it % C::kStages;
          if (!(ok = wait_bar(&bars->qd_full[s], (qd_it / C::kStages) & 1, abort_flag, a, 51))) break;
          tc_fence_after();
          issue_s(s);
          issue_dp(s);
          // K and V feed only the S^T and dP^T products: once the item's last
          // pair has completed, the next item's K/V copy may land.
          if (it.hi - it.lo == 1) mma_commit(&bars->kv_empty);
        }
        for (int i = it.lo; i < it.hi; ++i, ++qd_it) {
          const int s = qd_it % C::kStages;
          const bool more = i + 1 < it.hi;
          const int s1 = (qd_it + 1) % C::kStages;
          // the epilogue warpgroup has read the previous item's dV (dK below)
          if (i == it.lo && !(ok = wait_bar(&bars->dv_empty, (acc_cnt & 1) ^ 1, abort_flag, a, 52))) break;
          if (!(ok = wait_bar(&bars->p_ready, p_cnt & 1, abort_flag, a, 53))) break;
          ++p_cnt;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint64_t bd = sdesc_sw128(sDO(s) + kk * 16 * 128, kTile * 128, 1024);
            mma_ts(tmem + C::kDVCol, split_a(tmem + C::kSCol, kk), bd, idAcc, (kk > 0 || i > it.lo) ? 1u : 0u);
            // unnormalised pointwise: P^T's lo parts, 32 columns after the hi parts
            if constexpr (kHilo) mma_ts(tmem + C::kDVCol, split_a(tmem + C::kSCol + 32, kk), bd, idAcc, 1u);
          }
          if (!more) mma_commit(&bars->dv_full);  // the item's dV is complete
          if (more) {
            if (!(ok = wait_bar(&bars->qd_full[s1], ((qd_it + 1) / C::kStages) & 1, abort_flag, a, 54))) break;
            tc_fence_after();
            issue_s(s1);
          }
          if (i == it.lo && !(ok = wait_bar(&bars->dk_empty, (acc_cnt & 1) ^ 1, abort_flag, a, 56))) break;
          if (!(ok = wait_bar(&bars->ds_ready, ds_cnt & 1, abort_flag, a, 55))) break;
          ++ds_cnt;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint64_t bd = sdesc_sw128(sQ(s) + kk * 16 * 128, kTile * 128, 1024);
            mma_ts(tmem + C::kDKCol, split_a(tmem + C::kDPCol, kk), bd, idAcc, (kk > 0 || i > it.lo) ? 1u : 0u);
            // unnormalised pointwise: dS^T's lo parts
            if constexpr (kHilo) mma_ts(tmem + C::kDKCol, split_a(tmem + C::kDPCol + 32, kk), bd, idAcc, 1u);
          }
          mma_commit(&bars->qd_empty[s]);
          if (more) issue_dp(s1);
          if (i + 2 == it.hi) mma_commit(&bars->kv_empty);
        }
        if (!ok) break;
        mma_commit(&bars->dk_full);
        ++acc_cnt;
      }
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, a.timeout_ns);
    }
    __syncwarp();
  } else if (ACT == JATTN_SOFTMAX) {
    // ------------------------------------------------------------ LSE / Di staging (warps 2, 3)
    // Per step: -LSE log2(e) and -Di of the step's 128 query rows into one of
    // two shared-memory slots, a step ahead of the activation warpgroups, which
    // then only wait on the slot's barrier (bounded) and release it after
    // their dS. Rows past the sequence get 0 (their columns are masked).
    const int t = threadIdx.x - 64;  // 0 .. 63: rows t and t + 64 of each step
    uint32_t st = 0;
    bool ok = true;
    BwdItem it;
    for (long long r = 0; ok && load_bwd_item(a, r, it); ++r) {
      for (int i = it.lo; i < it.hi; ++i, ++st) {
        const int slot = st & 1;
        ok = __all_sync(0xffffffffu, wait_bar(&bars->ld_empty[slot], ((st >> 1) & 1) ^ 1, abort_flag, a, 65));
        if (!ok) break;
        float l2[2] = {0.0f, 0.0f}, dd[2] = {0.0f, 0.0f};
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {  // all four loads in flight before the stores
          const int iq = i * kTile + t + 64 * k2;
          if (iq < it.lq) {
            const int64_t gi = (it.q0 + iq) * a.H + it.h;
            l2[k2] = a.f0[gi] * kLog2e;
            dd[k2] = a.f1[gi];
          }
        }
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {  // stored negated: the activation adds them pairwise
          s_lse[slot * kTile + t + 64 * k2] = -l2[k2];
          s_di[slot * kTile + t + 64 * k2] = -dd[k2];
        }
        mbar_arrive(&bars->ld_full[slot]);
      }
    }
  }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kActRegs));
    const int g = (warp - 4) >> 2;                   // activation group: score columns [64g, 64g+64)
    const int row = 32 * (warp & 3) + lane;          // TMEM lane == key row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tSg = tmem + lane_base + C::kSCol + kCols * g;
    const uint32_t tDPg = tmem + lane_base + C::kDPCol + kCols * g;
    uint32_t s_cnt = 0, step = 0;
    BwdItem it, nit;
    bool have = load_bwd_item(a, 0, it), have_next = false;
    for (long long r = 0; have; ++r, it = nit, have = have_next) {
      have_next = load_bwd_item(a, r + 1, nit);
      const int jl = it.rt * kTile + row;  // sequence-local key row of this thread
      const bool valid = jl < it.lkv;
      const int delta = it.lkv - it.lq;
      int ilo, ihi;
      query_interval(jl, delta, it.lq, a.mask, a.window, ilo, ihi);
      if (!valid) ihi = ilo;  // rows past the sequence contribute nothing
      bool ok = true;
      for (int i = it.lo; i < it.hi; ++i, ++step) {
        float* lse_buf = s_lse + (step & 1) * kTile + kCols * g;
        float* di_buf = s_di + (step & 1) * kTile + kCols * g;
        if constexpr (ACT == JATTN_SOFTMAX) {  // this step's LSE / Di slot is filled
          ok = __all_sync(0xffffffffu, wait_bar(&bars->ld_full[step & 1], (step >> 1) & 1, abort_flag, a, 64));
          if (!ok) break;
        }
        ok = wait_bar(&bars->s_full, s_cnt & 1, abort_flag, a, 60);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float p[kCols];  // P^T (softmax) or act'(x) (pointwise) of this group's columns, fp32
        {
          uint32_t* pu = reinterpret_cast<uint32_t*>(p);
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c)
            tmem_ld32(tSg + c * 32, *reinterpret_cast<uint32_t(*)[32]>(pu + c * 32));
          tmem_ld_wait();
        }
        const int clo = ilo - i * kTile - kCols * g, chi = ihi - i * kTile - kCols * g;
        const bool edge = clo > 0 || chi < kCols;
        // 32-column chunks that no row of this warp sees (short or ragged query
        // tiles, masked corners) skip the arithmetic: their P and dS are zero.
        bool skip[kCols / 32];
#pragma unroll
        for (int k = 0; k < kCols / 32; ++k) skip[k] = __all_sync(0xffffffffu, max(clo, 32 * k) >= min(chi, 32 * k + 32));
        // chunks that every row of the warp sees whole need no per-element mask
        bool whole[kCols / 32];
#pragma unroll
        for (int k = 0; k < kCols / 32; ++k) whole[k] = __all_sync(0xffffffffu, clo <= 32 * k && chi >= 32 * k + 32);
        const uint64_t c2 = f2(a.scale_log2, a.scale_log2);
        const uint64_t* nlse2 = reinterpret_cast<const uint64_t*>(lse_buf);  // (-lse, -lse) pairs
        // P (and act' for the pointwise activations) of one 32-column chunk;
        // unnormalised pointwise: P's lo parts go to the group's other 32 S
        // columns (already read)
        auto chunk_p = [&](int c0, uint32_t(&pk)[16], auto masked) {
          ulonglong2 nl4;  // two (-lse, -lse) pairs per 16-byte shared load
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int c = c0 + e;
            float f0, f1;
            if constexpr (ACT == JATTN_SOFTMAX) {
              if ((e & 2) == 0) nl4 = reinterpret_cast<const ulonglong2*>(nlse2)[c / 4];
              float x0, x1;
              f2_split(ffma2(f2(p[c], p[c + 1]), c2, (e & 2) ? nl4.y : nl4.x), x0, x1);
              f0 = ex2_approx(x0);
              f1 = ex2_approx(x1);
              if constexpr (decltype(masked)::value) {
                f0 = (c >= clo && c < chi) ? f0 : 0.0f;
                f1 = (c + 1 >= clo && c + 1 < chi) ? f1 : 0.0f;
              }
              p[c] = f0;
              p[c + 1] = f1;
            } else {
              float g0, g1;
              act_and_grad<ACT>(p[c] * a.scale, f0, g0);
              act_and_grad<ACT>(p[c + 1] * a.scale, f1, g1);
              if (decltype(masked)::value && edge) {
                const bool a0 = c >= clo && c < chi, a1 = c + 1 >= clo && c + 1 < chi;
                f0 = a0 ? f0 : 0.0f;
                g0 = a0 ? g0 : 0.0f;
                f1 = a1 ? f1 : 0.0f;
                g1 = a1 ? g1 : 0.0f;
              }
              p[c] = g0;
              p[c + 1] = g1;
            }
            pk[e / 2] = pack_bf16x2(f0, f1);
            if constexpr (kHilo) tmem_st1(tSg + 32 + (c0 + e) / 2, bf16x2_lo(f0, f1, pk[e / 2]));
          }
        };
#pragma unroll
        for (int c0 = 0; c0 < kCols; c0 += 32) {
          uint32_t pk[16];
          if (skip[c0 / 32]) {
#pragma unroll
            for (int e = 0; e < 32; ++e) p[c0 + e] = 0.0f;
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = 0u;
            tmem_st16(tSg + c0 / 2, pk);
            if constexpr (kHilo) tmem_st16(tSg + 32 + c0 / 2, pk);
            continue;
          }
          // softmax: a second, unmasked copy for whole chunks; the longer pointwise
          // bodies keep one copy (two would crowd the instruction cache)
          if (ACT == JATTN_SOFTMAX && whole[c0 / 32])
            chunk_p(c0, pk, std::integral_constant<bool, ACT != JATTN_SOFTMAX>{});
          else
            chunk_p(c0, pk, std::true_type{});
          tmem_st16(tSg + c0 / 2, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_ready);

        ok = wait_bar(&bars->dp_full, s_cnt & 1, abort_flag, a, 61);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++s_cnt;
        tc_fence_after();
        {
          uint32_t dp[kCols];
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c) tmem_ld32(tDPg + c * 32, *reinterpret_cast<uint32_t(*)[32]>(dp + c * 32));
          tmem_ld_wait();
#pragma unroll
          for (int c0 = 0; c0 < kCols; c0 += 32) {
            uint32_t pk[16];
            if (skip[c0 / 32]) {
#pragma unroll
              for (int e = 0; e < 16; ++e) pk[e] = 0u;
              tmem_st16(tDPg + c0 / 2, pk);
              if constexpr (kHilo) tmem_st16(tDPg + 32 + c0 / 2, pk);
              continue;
            }
            ulonglong2 nd4;  // two (-Di, -Di) pairs per 16-byte shared load
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int c = c0 + e;
              float d0, d1;
              if constexpr (ACT == JATTN_SOFTMAX) {
                if ((e & 2) == 0) nd4 = reinterpret_cast<const ulonglong2*>(di_buf)[c / 4];
                const uint64_t ndi2 = (e & 2) ? nd4.y : nd4.x;
                f2_split(fmul2(f2(p[c], p[c + 1]),
                               fadd2(f2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), ndi2)), d0, d1);
                pk[e / 2] = pack_bf16x2(d0, d1);
              } else {
                d0 = p[c] * __uint_as_float(dp[c]);
                d1 = p[c + 1] * __uint_as_float(dp[c + 1]);
                pk[e / 2] = pack_bf16x2(d0, d1);
                // unnormalised: dS's lo parts in the group's other 32 dP columns (already read)
                if constexpr (kHilo) tmem_st1(tDPg + 32 + (c0 + e) / 2, bf16x2_lo(d0, d1, pk[e / 2]));
              }
            }
            tmem_st16(tDPg + c0 / 2, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->ds_ready);
        if constexpr (ACT == JATTN_SOFTMAX) mbar_arrive(&bars->ld_empty[step & 1]);
      }
      if (!ok) break;
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
    // ------------------------------------------------------------ epilogue warpgroup (warps 12-15)
    // Drains each item's dV and dK while the activation warpgroups start the
    // next item; items that no query sees get zero rows.
    const int row = 32 * (warp & 3) + lane;  // TMEM lane == key row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    uint32_t acc_cnt = 0;
    BwdItem it;
    for (long long r = 0; load_bwd_item(a, r, it); ++r) {
      const int jl = it.rt * kTile + row;
      const bool valid = jl < it.lkv;
      const int64_t gk = it.k0 + jl;
      __nv_bfloat16* dv_row = a.out1 + (gk * a.H + it.h) * D;
      __nv_bfloat16* dk_row = a.out0 + (gk * a.H + it.h) * D;
      if (it.hi <= it.lo) {
        if (valid) {
          zero_row(dv_row, D);
          zero_row(dk_row, D);
        }
        continue;
      }
      const float cn = (ACT != JATTN_SOFTMAX && a.norm_by_lkv && it.lkv > 0) ? 1.0f / it.lkv : 1.0f;
      if (!__all_sync(0xffffffffu, wait_bar(&bars->dv_full, acc_cnt & 1, abort_flag, a, 62))) break;
      tc_fence_after();
      epi_rows<D>(tmem + lane_base + C::kDVCol, cn, dv_row, valid, &bars->dv_empty, a, nullptr, nullptr);
      const float* rc = nullptr;  // rotary backward of dK
      const float* rs = nullptr;
      if (valid) rope_rows_at(a, rope_pos_k(jl, it.lkv - it.lq), rc, rs);
      if (!__all_sync(0xffffffffu, wait_bar(&bars->dk_full, acc_cnt & 1, abort_flag, a, 66))) break;
      ++acc_cnt;
      tc_fence_after();
      epi_rows<D>(tmem + lane_base + C::kDKCol, cn * a.scale, dk_row, valid, &bars->dk_empty, a, rc, rs);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------- dQ
// Two layouts of the K / V tiles, picked per call (dq_split_rings in the
// host code) from the key tiles an item holds on average:
//   one ring (SPLIT = false): stage s holds K(j) and V(j), one barrier and one
//     release per tile for the MMA issuer; the softmax Di warps also get the
//     item's O tile in shared memory;
//   two rings (SPLIT = true): K tiles, needed first (by S, a tile ahead) and
//     read last (by dQ), in a deeper ring than V tiles (read by dP only). With
//     one two-stage ring each K copy could only start once dQ had read the
//     tile two before, so long items saw its latency on every tile; items of
//     few tiles pay more for the extra barrier and release than they gain.
//     The Di warps read O from global memory (prefetched into L2).
template <int D, bool SPLIT>
struct DqCfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kKStages = SPLIT ? 3 : ((D == 128) ? 2 : 3);
  static constexpr int kVStages = SPLIT ? ((D == 128) ? 2 : 3) : kKStages;
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = kTileBytes;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kKStride = SPLIT ? kTileBytes : 2 * kTileBytes;  // K stage s at kKOff + s strides
  static constexpr int kVOff = SPLIT ? kKOff + kKStages * kTileBytes : kKOff + kTileBytes;
  static constexpr int kVStride = kKStride;                             // V stage s at kVOff + s strides
  static constexpr int kBarOff = SPLIT ? kVOff + kVStages * kTileBytes : kKOff + kKStages * 2 * kTileBytes;
  // [2][128] Di, then [2][128] LSE, handed to the activation warpgroups
  // (softmax), then the two barriers that publish a slot's LSE ahead of its Di
  static constexpr int kDiOff = kBarOff + 256;
  static constexpr int kLseBarOff = kDiOff + 4 * kTile * 4;
  static constexpr int kOOff = (kLseBarOff + 16 + 1023) / 1024 * 1024;  // O tile (one ring, softmax)
  static constexpr int kSmemBytes = SPLIT ? kLseBarOff + 16 : kOOff + kTileBytes;  // base 1024-aligned
  static constexpr uint32_t kSCol = 0, kDPCol = 256, kDQCol = 384;  // S double-buffered at 0 and 128
};

struct DqBars {
  uint64_t qd_full, qd_empty;
  uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
  uint64_t s_full[2], dp_full, ds_ready, acc_full, acc_empty;
  uint64_t di_full[2], di_empty[2];  // Di slots (softmax)
  uint64_t ot_full, ot_empty;         // O tile for Di (one ring, softmax)
  uint64_t xbar[4];                   // per lane quarter: row exchange between the activation groups, 64 arrivals
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

static_assert(sizeof(DqBars) <= 256, "barrier block overflows its slot");
static_assert(DqCfg<128, false>::kSmemBytes <= 227 * 1024 && DqCfg<64, false>::kSmemBytes <= 227 * 1024 &&
                  DqCfg<128, true>::kSmemBytes <= 227 * 1024 && DqCfg<64, true>::kSmemBytes <= 227 * 1024,
              "shared memory");

template <int D, int ACT, bool IN_TILE, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmO, const AttnArgs a) {
  using C = DqCfg<D, SPLIT>;
  constexpr bool kOTile = ACT == JATTN_SOFTMAX && !IN_TILE && !SPLIT;  // Di from an O tile in shared memory
  constexpr bool kHilo = JATTN_HILO && ACT != JATTN_SOFTMAX;  // dS as bf16 hi + lo parts
  // IN_TILE (softmax, a.in_tile_stats): statistics and Di from the single key
  // tile of every item, compiled apart so the general path carries none of it
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned tiles and no slack for realigning: a misaligned base is an error
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(a.status, JATTN_ERR_UNSUPPORTED, 19, blockIdx.x);
    return;
  }
  uint8_t* sm = smem_raw;
  DqBars* bars = reinterpret_cast<DqBars*>(sm + C::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&bars->qd_full, 1);
    // softmax: the Di warps read dO from this buffer too, so they also release it
    mbar_init(&bars->qd_empty, (ACT == JATTN_SOFTMAX && !IN_TILE) ? 1 + 64 : 1);
    for (int x = 0; x < 4; ++x) mbar_init(&bars->xbar[x], 64);
    mbar_init(&bars->ot_full, 1);
    mbar_init(&bars->ot_empty, 64);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->ds_ready, kNG * kTile);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, kTile);  // the epilogue warpgroup's threads
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(&bars->di_full[s2], 64);
      mbar_init(reinterpret_cast<uint64_t*>(sm + C::kLseBarOff) + s2, 64);
      mbar_init(&bars->di_empty[s2], kNG * kTile);
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
    if (lane == 0) {
      uint32_t item_cnt = 0, kv_it = 0;
      bool q_armed = false, ok = true;
      BwdItem it, nit;
      bool have = load_bwd_item(a, 0, it), have_next = false;
      for (long long r = 0; have && ok; ++r, it = nit, have = have_next) {
        have_next = load_bwd_item(a, r + 1, nit);
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->qd_empty, (item_cnt & 1) ^ 1, abort_flag, a, 70))) break;
        ++item_cnt;
        const int yq = static_cast<int>(it.q0) + it.rt * kTile;
        if (!(a.debug_flags & 1)) {
          mbar_arrive_expect_tx(&bars->qd_full, 2 * C::kTileBytes);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(sm + C::kQOff + c * kTile * 128, &tmQ, &bars->qd_full, it.h * D + c * 64, yq);
            tma_load_2d(sm + C::kDOOff + c * kTile * 128, &tmDO, &bars->qd_full, it.h * D + c * 64, yq);
          }
          q_armed = true;
          if constexpr (kOTile) {  // O tile for the Di warps
            if (!(ok = wait_bar(&bars->ot_empty, ((item_cnt - 1) & 1) ^ 1, abort_flag, a, 74))) break;
            mbar_arrive_expect_tx(&bars->ot_full, C::kTileBytes);
            for (int c = 0; c < D / 64; ++c)
              tma_load_2d(sm + C::kOOff + c * kTile * 128, &tmO, &bars->ot_full, it.h * D + c * 64, yq);
          }
        }
        for (int j = it.lo; j < it.hi; ++j, ++kv_it) {
          const int sk = kv_it % C::kKStages, sv = kv_it % C::kVStages;
          const int yk = static_cast<int>(it.k0) + j * kTile;
          if (!(ok = wait_bar(&bars->k_empty[sk], ((kv_it / C::kKStages) & 1) ^ 1, abort_flag, a, 71))) break;
          mbar_arrive_expect_tx(&bars->k_full[sk], (SPLIT ? 1 : 2) * C::kTileBytes);
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(sm + C::kKOff + sk * C::kKStride + c * kTile * 128, &tmK, &bars->k_full[sk],
                        it.h * D + c * 64, yk);
          uint64_t* vbar = &bars->k_full[sk];  // one ring: V lands on its stage's barrier
          if constexpr (SPLIT) {
            if (!(ok = wait_bar(&bars->v_empty[sv], ((kv_it / C::kVStages) & 1) ^ 1, abort_flag, a, 72))) break;
            vbar = &bars->v_full[sv];
            mbar_arrive_expect_tx(vbar, C::kTileBytes);
          }
          for (int c = 0; c < D / 64; ++c)
            tma_load_2d(sm + C::kVOff + sv * C::kVStride + c * kTile * 128, &tmV, vbar, it.h * D + c * 64, yk);
        }
      }
      if (q_armed) drain_wait(&bars->qd_full, (item_cnt - 1) & 1, a.timeout_ns);
      if (q_armed && kOTile) drain_wait(&bars->ot_full, (item_cnt - 1) & 1, a.timeout_ns);
      for (uint32_t i = (kv_it > (uint32_t)C::kKStages ? kv_it - C::kKStages : 0); i < kv_it; ++i)
        drain_wait(&bars->k_full[i % C::kKStages], (i / C::kKStages) & 1, a.timeout_ns);
      if (SPLIT)
        for (uint32_t i = (kv_it > (uint32_t)C::kVStages ? kv_it - C::kVStages : 0); i < kv_it; ++i)
          drain_wait(&bars->v_full[i % C::kVStages], (i / C::kVStages) & 1, a.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kTile, kTile, false, false);
      constexpr uint32_t idAcc = idesc_bf16_f32(kTile, D, false, true);
      const uint32_t sQ = smem_u32(sm + C::kQOff), sDO = smem_u32(sm + C::kDOOff);
      const uint32_t sK0 = smem_u32(sm + C::kKOff), sV0 = smem_u32(sm + C::kVOff);
      uint32_t item_cnt = 0, kv_it = 0, ds_cnt = 0, acc_cnt = 0, step = 0;
      bool ok = true;
      auto sK = [&](int s) { return sK0 + s * C::kKStride; };
      auto sV = [&](int s) { return sV0 + s * C::kVStride; };
      // the V tile of global tile t is present (two rings: its own barrier;
      // one ring: the stage's barrier, already waited for S)
      auto wait_v = [&](uint32_t t) {
        if constexpr (SPLIT) {
          if (!wait_bar(&bars->v_full[t % C::kVStages], (t / C::kVStages) & 1, abort_flag, a, 86)) return false;
          tc_fence_after();
        }
        return true;
      };
      auto kmajor = [](uint32_t base, int kk) {
        return sdesc_sw128(base + (kk >> 2) * (kTile * 128) + (kk & 3) * 32, 16, 1024);
      };
      auto issue_s = [&](int s, uint32_t st) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::kSCol + (st & 1) * kTile, kmajor(sQ, kk), kmajor(sK(s), kk), idS, kk > 0);
        mma_commit(&bars->s_full[st & 1]);
      };
      auto issue_dp = [&](int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + C::kDPCol, kmajor(sDO, kk), kmajor(sV(s), kk), idS, kk > 0);
        mma_commit(&bars->dp_full);
        if constexpr (SPLIT) mma_commit(&bars->v_empty[s]);  // V(j) feeds dP(j) only
      };
      BwdItem it, nit;
      bool have = load_bwd_item(a, 0, it), have_next = false;
      for (long long r = 0; have && ok; ++r, it = nit, have = have_next) {
        have_next = load_bwd_item(a, r + 1, nit);
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->qd_full, item_cnt & 1, abort_flag, a, 80))) break;
        ++item_cnt;
        tc_fence_after();
        {
          const int sk = kv_it % C::kKStages, sv = kv_it % C::kVStages;
          if (!(ok = wait_bar(&bars->k_full[sk], (kv_it / C::kKStages) & 1, abort_flag, a, 81))) break;
          tc_fence_after();
          issue_s(sk, step);
          if (!(ok = wait_v(kv_it))) break;
          issue_dp(sv);
          // Q and dO feed only the S and dP products: once the item's last pair
          // has completed, the next item's Q/dO copy may land.
          if (it.hi - it.lo == 1) mma_commit(&bars->qd_empty);
        }
        for (int j = it.lo; j < it.hi; ++j, ++kv_it, ++step) {
          const int s = kv_it % C::kKStages;
          const bool more = j + 1 < it.hi;
          const uint32_t k1 = kv_it + 1;
          if (more) {
            if (!(ok = wait_bar(&bars->k_full[k1 % C::kKStages], (k1 / C::kKStages) & 1, abort_flag, a, 82))) break;
            tc_fence_after();
            issue_s(k1 % C::kKStages, step + 1);
          }
          if (j == it.lo) {
            if (!(ok = wait_bar(&bars->acc_empty, (acc_cnt & 1) ^ 1, abort_flag, a, 83))) break;
          }
          if (!(ok = wait_bar(&bars->ds_ready, ds_cnt & 1, abort_flag, a, 84))) break;
          ++ds_cnt;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint64_t bd = sdesc_sw128(sK(s) + kk * 16 * 128, kTile * 128, 1024);
            mma_ts(tmem + C::kDQCol, split_a(tmem + C::kDPCol, kk), bd, idAcc, (kk > 0 || j > it.lo) ? 1u : 0u);
            // unnormalised pointwise: dS's lo parts, 32 columns after the hi parts
            if constexpr (kHilo) mma_ts(tmem + C::kDQCol, split_a(tmem + C::kDPCol + 32, kk), bd, idAcc, 1u);
          }
          mma_commit(&bars->k_empty[s]);  // K(j) was read by S(j) and, last, by dQ(j)
          if (more) {
            if (!(ok = wait_v(k1))) break;
            issue_dp(k1 % C::kVStages);
          }
          if (j + 2 == it.hi) mma_commit(&bars->qd_empty);
        }
        if (!ok) break;
        mma_commit(&bars->acc_full);
        ++acc_cnt;
      }
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, a.timeout_ns);
    }
    __syncwarp();
  } else if (ACT == JATTN_SOFTMAX && !IN_TILE) {
    // ------------------------------------------------------------ Di warps (2, 3)
    // Di = rowsum(dO * O) for each item's 128 query rows, from the dO tile the
    // producer loaded for the MMAs and O (one ring: a tile the producer loads
    // for this purpose; two rings: the rows in global memory, a.in0, with a
    // prefetch into L2 before the waits): into a shared-memory slot for the
    // activation warpgroups and to global memory for the dK/dV pass, which
    // runs after this one. The same slot carries each row's LSE, loaded here,
    // off the activation warps' critical path. Items with a single key tile
    // get an exact Di from the activation warps instead (sum of P * dP over
    // the tile), so here they only pass the LSE. Lane l of warp 2 + w owns tile
    // rows 64w + l and 64w + 32 + l; walking a row's 16-byte pieces of the
    // 128-byte-swizzled tiles in swizzled order spreads the lanes over the
    // banks (the O tile shares the layout, so the same addresses pair columns).
    const int dw = warp - 2;
    float* di_s = reinterpret_cast<float*>(sm + C::kDiOff);
    const uint32_t sDO = smem_u32(sm + C::kDOOff);
    const uint32_t sO = smem_u32(sm + (kOTile ? C::kOOff : 0));
    uint32_t n_item = 0;
    BwdItem it;
    for (long long r = 0; load_bwd_item(a, r, it); ++r) {
      if (it.hi <= it.lo) continue;  // no Q/dO/O copy for it, and nothing reads its Di
      const int slot = n_item & 1;
      const bool single = it.hi - it.lo == 1;
      int rl[2];
      bool dot[2];
      float lse_rows[2], acc[2] = {0.0f, 0.0f};
      const uint4* orow[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        rl[h2] = 64 * dw + 32 * h2 + lane;
        const int il = it.rt * kTile + rl[h2];
        const int64_t gi = (it.q0 + il) * a.H + it.h;
        dot[h2] = il < it.lq && !single;  // rows past the sequence: their Di is never read
        orow[h2] = reinterpret_cast<const uint4*>(a.in0 + gi * D);
        lse_rows[h2] = (il < it.lq) ? a.f0[gi] : 0.0f;
      }
      if constexpr (!kOTile) {  // both rows of O on their way into L2 while the waits below pass
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
          if (dot[h2])
#pragma unroll
            for (int line = 0; line < D * 2 / 128; ++line)
              asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(orow[h2]) + 128 * line));
      }
      bool ok = wait_bar(&bars->di_empty[slot], ((n_item >> 1) & 1) ^ 1, abort_flag, a, 75);
      if (!__all_sync(0xffffffffu, ok)) break;
      // the rows' LSE first: the activation warps need it for P, Di only for dS
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) di_s[(2 + slot) * kTile + rl[h2]] = lse_rows[h2];
      mbar_arrive(reinterpret_cast<uint64_t*>(sm + C::kLseBarOff) + slot);
      ok = wait_bar(&bars->qd_full, n_item & 1, abort_flag, a, 76);
      if (kOTile) ok = ok && wait_bar(&bars->ot_full, n_item & 1, abort_flag, a, 77);
      if (!__all_sync(0xffffffffu, ok)) break;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
        for (int cb = 0; cb < (single ? 0 : D / 64); ++cb) {
          uint4 ov[8];  // 64 columns of O, loaded before the dot product
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            if constexpr (kOTile) {
              const uint32_t off = cb * (kTile * 128) + rl[h2] * 128 + ((ch ^ (rl[h2] & 7)) << 4);
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(ov[ch].x), "=r"(ov[ch].y), "=r"(ov[ch].z), "=r"(ov[ch].w)
                           : "r"(sO + off));
            } else {
              ov[ch] = dot[h2] ? __ldg(orow[h2] + 8 * cb + ch) : make_uint4(0, 0, 0, 0);
            }
          }
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint32_t off = cb * (kTile * 128) + rl[h2] * 128 + ((ch ^ (rl[h2] & 7)) << 4);
            const uint32_t x[4] = {ov[ch].x, ov[ch].y, ov[ch].z, ov[ch].w};
            uint32_t y[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(y[0]), "=r"(y[1]), "=r"(y[2]), "=r"(y[3])
                         : "r"(sDO + off));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x[e]));
              const float2 yf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y[e]));
              acc[h2] = fmaf(xf.x, yf.x, fmaf(xf.y, yf.y, acc[h2]));
            }
          }
        }
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        di_s[slot * kTile + rl[h2]] = acc[h2];
        if (dot[h2]) a.f1[(it.q0 + it.rt * kTile + rl[h2]) * a.H + it.h] = acc[h2];
      }
      mbar_arrive(&bars->di_full[slot]);
      if constexpr (kOTile) mbar_arrive(&bars->ot_empty);
      mbar_arrive(&bars->qd_empty);
      ++n_item;
    }
  }
  } else if (warp < 12) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kActRegs));
    const int g = (warp - 4) >> 2;                  // activation group: score columns [64g, 64g+64)
    const int row = 32 * (warp & 3) + lane;         // TMEM lane == query row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tDPg = tmem + lane_base + C::kDPCol + kCols * g;
    const int quarter = warp & 3;
    uint32_t step = 0, dp_cnt = 0, di_item = 0, x_cnt = 0;
    // Row exchange with the partner warp of the other group (same TMEM lanes):
    // each writes its value into column k of its own half of the current S
    // buffer, whose scores it has already read, they meet on the quarter's
    // mbarrier (bounded wait), and each reads the partner's column. The S
    // buffer is not rewritten before this step's dS is handed over.
    auto exchange = [&](float v, int k, uint32_t sbuf, bool& okx) -> float {
      const uint32_t col = tmem + lane_base + C::kSCol + sbuf * kTile + k;
      tmem_st1(col + kCols * g, __float_as_uint(v));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->xbar[quarter]);
      okx = __all_sync(0xffffffffu, wait_bar(&bars->xbar[quarter], x_cnt & 1, abort_flag, a, 95));
      ++x_cnt;
      if (!okx) return 0.0f;
      tc_fence_after();
      const float r = __uint_as_float(tmem_ld1(col + kCols * (g ^ 1)));
      tmem_ld_wait();
      return r;
    };
    BwdItem it, nit;
    bool have = load_bwd_item(a, 0, it), have_next = false;
    for (long long r = 0; have; ++r, it = nit, have = have_next) {
      have_next = load_bwd_item(a, r + 1, nit);
      const int il = it.rt * kTile + row;
      const bool valid = il < it.lq;
      const int delta = it.lkv - it.lq;
      int klo, khi;
      key_interval(il, delta, it.lkv, a.mask, a.window, klo, khi);
      if (!valid) khi = klo;
      const int64_t gi = (it.q0 + il) * a.H + it.h;
      float lse2 = 0.0f, di = 0.0f;
      const bool single = it.hi - it.lo == 1;  // softmax: Di (and with in-tile stats, LSE) from the tile
      // softmax: the Di slot whose Di this item still has to read before its
      // first dS (the LSE, needed for P, is read here)
      int di_slot = -1;
      uint32_t di_par = 0;
      const float* di_s = reinterpret_cast<const float*>(sm + C::kDiOff);
      if constexpr (ACT == JATTN_SOFTMAX) {
        if (it.hi > it.lo && !IN_TILE) {  // items without a key tile use no Di and get no slot
          const int slot = di_item & 1;
          bool okd = wait_bar(reinterpret_cast<uint64_t*>(sm + C::kLseBarOff) + slot, (di_item >> 1) & 1, abort_flag,
                              a, 94);
          if (!__all_sync(0xffffffffu, okd)) break;
          const float lse_row = di_s[(2 + slot) * kTile + row];
          if (valid && khi > klo) lse2 = lse_row * kLog2e;
          if (single) {
            mbar_arrive(&bars->di_empty[slot]);  // Di comes from the tile itself
          } else {
            di_slot = slot;
            di_par = (di_item >> 1) & 1;
          }
          ++di_item;
        }
      }
      bool ok = true;
      for (int j = it.lo; j < it.hi; ++j, ++step) {
        ok = wait_bar(&bars->s_full[step & 1], (step >> 1) & 1, abort_flag, a, 90);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float p[kCols];
        {
          uint32_t* pu = reinterpret_cast<uint32_t*>(p);
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c)
            tmem_ld32(tmem + lane_base + C::kSCol + (step & 1) * kTile + kCols * g + c * 32,
                      *reinterpret_cast<uint32_t(*)[32]>(pu + c * 32));
          tmem_ld_wait();
        }
        const int clo = klo - j * kTile - kCols * g, chi = khi - j * kTile - kCols * g;
        const bool edge = clo > 0 || chi < kCols;
        // 32-column chunks that no row of this warp sees (rows past a short query
        // tile, masked corners) skip the arithmetic: their dS is zero.
        bool skip[kCols / 32];
#pragma unroll
        for (int k = 0; k < kCols / 32; ++k) skip[k] = __all_sync(0xffffffffu, max(clo, 32 * k) >= min(chi, 32 * k + 32));
        // chunks that every row of the warp sees whole need no per-element mask
        bool whole[kCols / 32];
#pragma unroll
        for (int k = 0; k < kCols / 32; ++k) whole[k] = __all_sync(0xffffffffu, clo <= 32 * k && chi >= 32 * k + 32);
        const uint64_t c2 = f2(a.scale_log2, a.scale_log2), nl2 = f2(-lse2, -lse2);
        const uint32_t sbuf = step & 1;
        float row_lse = -INFINITY;  // in-tile statistics: natural-log LSE of this row
        auto chunk_p = [&](int c0, auto masked) {
#pragma unroll
          for (int c = c0; c < c0 + 32; c += 2) {
            float v0, v1;
            if constexpr (ACT == JATTN_SOFTMAX) {
              float x0, x1;
              f2_split(ffma2(f2(p[c], p[c + 1]), c2, nl2), x0, x1);
              v0 = ex2_approx(x0);
              v1 = ex2_approx(x1);
            } else {
              float f;
              act_and_grad<ACT>(p[c] * a.scale, f, v0);
              act_and_grad<ACT>(p[c + 1] * a.scale, f, v1);
            }
            if (decltype(masked)::value && (ACT == JATTN_SOFTMAX || edge)) {
              v0 = (c >= clo && c < chi) ? v0 : 0.0f;
              v1 = (c + 1 >= clo && c + 1 < chi) ? v1 : 0.0f;
            }
            p[c] = v0;
            p[c + 1] = v1;
          }
        };
        if (ACT == JATTN_SOFTMAX && IN_TILE) {
          // the row's whole key range lies in this tile: its maximum and sum
          // come from the two groups' halves, P = exp(s - m) / l exactly
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < kCols; ++c) {
            const float v = (c >= clo && c < chi) ? p[c] : -INFINITY;
            p[c] = v;
            mx = fmaxf(mx, v);
          }
          mx = fmaxf(mx, exchange(mx, 0, sbuf, ok));
          if (!ok) break;
          const float mref = (mx == -INFINITY) ? 0.0f : mx * a.scale_log2;
          float l = 0.0f;
#pragma unroll
          for (int c = 0; c < kCols; ++c) {
            p[c] = ex2_approx(fmaf(p[c], a.scale_log2, -mref));
            l += p[c];
          }
          l += exchange(l, 1, sbuf, ok);
          if (!ok) break;
          const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
#pragma unroll
          for (int c = 0; c < kCols; ++c) p[c] *= inv;
          row_lse = (l > 0.0f) ? (mref + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        } else {
#pragma unroll
          for (int c0 = 0; c0 < kCols; c0 += 32) {
            if (skip[c0 / 32]) continue;
            // softmax: a second, unmasked copy for whole chunks; the longer pointwise
            // bodies keep one copy (two would crowd the instruction cache)
            if (ACT == JATTN_SOFTMAX && whole[c0 / 32])
              chunk_p(c0, std::integral_constant<bool, ACT != JATTN_SOFTMAX>{});
            else
              chunk_p(c0, std::true_type{});
          }
        }
        ok = wait_bar(&bars->dp_full, dp_cnt & 1, abort_flag, a, 91);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++dp_cnt;
        tc_fence_after();
        {
          uint32_t dp[kCols];
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c) tmem_ld32(tDPg + c * 32, *reinterpret_cast<uint32_t(*)[32]>(dp + c * 32));
          tmem_ld_wait();
          if (ACT == JATTN_SOFTMAX && !IN_TILE && di_slot >= 0) {  // the item's first dS: its Di
            ok = __all_sync(0xffffffffu, wait_bar(&bars->di_full[di_slot], di_par, abort_flag, a, 96));
            if (!ok) break;
            const float di_row = di_s[di_slot * kTile + row];
            if (valid && khi > klo) di = di_row;
            mbar_arrive(&bars->di_empty[di_slot]);
            di_slot = -1;
          }
          if (ACT == JATTN_SOFTMAX && single) {
            // Di = sum_j P_ij dP_ij over the row's whole key range, in fp32: exact
            // where a Di from the stored bf16 O would carry O's rounding (rows that
            // see a few keys, where that rounding is large next to dQ)
            float part = 0.0f;
#pragma unroll
            for (int k = 0; k < kCols / 32; ++k) {
              if (skip[k] && !IN_TILE) continue;  // chunk not computed: P is zero there
#pragma unroll
              for (int c = 32 * k; c < 32 * k + 32; ++c) part = fmaf(p[c], __uint_as_float(dp[c]), part);
            }
            di = part + exchange(part, 2, sbuf, ok);
            if (!ok) break;
            if (g == 0 && valid) {
              a.f1[gi] = di;
              if (IN_TILE) a.f0[gi] = row_lse;
            }
          }
          const uint64_t ndi2 = f2(-di, -di);
#pragma unroll
          for (int c0 = 0; c0 < kCols; c0 += 32) {
            uint32_t pk[16];
            if (skip[c0 / 32]) {
#pragma unroll
              for (int e = 0; e < 16; ++e) pk[e] = 0u;
              tmem_st16(tDPg + c0 / 2, pk);
              if constexpr (kHilo) tmem_st16(tDPg + 32 + c0 / 2, pk);
              continue;
            }
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int c = c0 + e;
              float d0, d1;
              if constexpr (ACT == JATTN_SOFTMAX) {
                f2_split(fmul2(f2(p[c], p[c + 1]),
                               fadd2(f2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])), ndi2)), d0, d1);
                pk[e / 2] = pack_bf16x2(d0, d1);
              } else {
                d0 = p[c] * __uint_as_float(dp[c]);
                d1 = p[c + 1] * __uint_as_float(dp[c + 1]);
                pk[e / 2] = pack_bf16x2(d0, d1);
                // unnormalised: dS's lo parts in the group's other 32 dP columns (already read)
                if constexpr (kHilo) tmem_st1(tDPg + 32 + (c0 + e) / 2, bf16x2_lo(d0, d1, pk[e / 2]));
              }
            }
            tmem_st16(tDPg + c0 / 2, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->ds_ready);
      }
      if (!ok) break;
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
    // ------------------------------------------------------------ epilogue warpgroup (warps 12-15)
    // Drains each item's dQ (one row per thread, rotated back when asked)
    // while the activation warpgroups start the next item; rows that see no
    // key get zeros (and, with in-tile statistics, LSE = -inf and Di = 0).
    const int row = 32 * (warp & 3) + lane;  // TMEM lane == query row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    uint32_t acc_cnt = 0;
    BwdItem it;
    for (long long r = 0; load_bwd_item(a, r, it); ++r) {
      const int il = it.rt * kTile + row;
      const bool valid = il < it.lq;
      const int64_t gi = (it.q0 + il) * a.H + it.h;
      __nv_bfloat16* dq_row = a.out0 + gi * D;
      if (it.hi <= it.lo) {
        if (valid) {
          zero_row(dq_row, D);
          if (ACT == JATTN_SOFTMAX && IN_TILE) {
            a.f0[gi] = -INFINITY;
            a.f1[gi] = 0.0f;
          }
        }
        continue;
      }
      const float cn = (ACT != JATTN_SOFTMAX && a.norm_by_lkv && it.lkv > 0) ? 1.0f / it.lkv : 1.0f;
      const float* rc = nullptr;  // rotary backward of dQ
      const float* rs = nullptr;
      if (valid) rope_rows_at(a, rope_pos_q(il, it.lkv - it.lq), rc, rs);
      if (!__all_sync(0xffffffffu, wait_bar(&bars->acc_full, acc_cnt & 1, abort_flag, a, 92))) break;
      ++acc_cnt;
      tc_fence_after();
      epi_rows<D>(tmem + lane_base + C::kDQCol, cn * a.scale, dq_row, valid, &bars->acc_empty, a, rc, rs);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <typename K>
cudaError_t launch5(K kern, int smem, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                    const CUtensorMap& dout, const CUtensorMap& o, const AttnArgs& a, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(q, k, v, dout, o, a);
  return cudaGetLastError();
}

// dQ kernel of one activation and head dimension, in the chosen K / V layout
// (two rings only at D = 128, where one ring holds two stages).
template <int D, int ACT, bool IN_TILE>
cudaError_t launch_dq_layout(bool split, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const CUtensorMap& dout, const CUtensorMap& o, const AttnArgs& a, int grid,
                             cudaStream_t stream) {
  if constexpr (D == 128 && !IN_TILE) {
    if (split)
      return launch5(dq_kernel<D, ACT, IN_TILE, true>, DqCfg<D, true>::kSmemBytes, q, k, v, dout, o, a, grid, stream);
  }
  // the O tile only for softmax's Di warps (the rest of the on-chip memory stays L1)
  constexpr int smem = (ACT == JATTN_SOFTMAX && !IN_TILE) ? DqCfg<D, false>::kSmemBytes : DqCfg<D, false>::kOOff;
  return launch5(dq_kernel<D, ACT, IN_TILE, false>, smem, q, k, v, dout, o, a, grid, stream);
}

template <typename K>
cudaError_t launch4(K kern, int smem, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                    const CUtensorMap& dout, const AttnArgs& a, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(q, k, v, dout, a);
  return cudaGetLastError();
}

}  // namespace

#if JATTN_HILO
cudaError_t launch_bwd_dkdv_hilo(int D, int act, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& dout, const AttnArgs& a, int grid,
                                 cudaStream_t stream) {
#else
cudaError_t launch_bwd_dkdv(int D, int act, bool hilo, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, const CUtensorMap& dout, const AttnArgs& a, int grid,
                            cudaStream_t stream) {
  if (hilo && act != JATTN_SOFTMAX) return launch_bwd_dkdv_hilo(D, act, q, k, v, dout, a, grid, stream);
  if (act == JATTN_SOFTMAX)
    return D == 128 ? launch4(dkdv_kernel<128, JATTN_SOFTMAX>, DkdvCfg<128>::kSmemBytes, q, k, v, dout, a,
                              grid, stream)
                    : launch4(dkdv_kernel<64, JATTN_SOFTMAX>, DkdvCfg<64>::kSmemBytes, q, k, v, dout, a, grid,
                              stream);
#endif
  if (D == 128) {
    constexpr int sm = DkdvCfg<128>::kSmemBytes;
    if (act == JATTN_SILU) return launch4(dkdv_kernel<128, JATTN_SILU>, sm, q, k, v, dout, a, grid, stream);
    if (act == JATTN_GELU_POLY)
      return launch4(dkdv_kernel<128, JATTN_GELU_POLY>, sm, q, k, v, dout, a, grid, stream);
    if (act == JATTN_GELU_TANH)
      return launch4(dkdv_kernel<128, JATTN_GELU_TANH>, sm, q, k, v, dout, a, grid, stream);
    return cudaErrorInvalidValue;
  }
  constexpr int sm = DkdvCfg<64>::kSmemBytes;
  if (act == JATTN_SILU) return launch4(dkdv_kernel<64, JATTN_SILU>, sm, q, k, v, dout, a, grid, stream);
  if (act == JATTN_GELU_POLY) return launch4(dkdv_kernel<64, JATTN_GELU_POLY>, sm, q, k, v, dout, a, grid, stream);
  if (act == JATTN_GELU_TANH) return launch4(dkdv_kernel<64, JATTN_GELU_TANH>, sm, q, k, v, dout, a, grid, stream);
  return cudaErrorInvalidValue;
}

#if JATTN_HILO
cudaError_t launch_bwd_dq_hilo(int D, int act, bool split, const CUtensorMap& q, const CUtensorMap& k,
                               const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& o, const AttnArgs& a,
                               int grid, cudaStream_t stream) {
#else
cudaError_t launch_bwd_dq(int D, int act, bool hilo, bool split, const CUtensorMap& q, const CUtensorMap& k,
                          const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& o, const AttnArgs& a,
                          int grid, cudaStream_t stream) {
  if (hilo && act != JATTN_SOFTMAX) return launch_bwd_dq_hilo(D, act, split, q, k, v, dout, o, a, grid, stream);
  if (act == JATTN_SOFTMAX) {
    if (a.in_tile_stats)
      return D == 128 ? launch_dq_layout<128, JATTN_SOFTMAX, true>(false, q, k, v, dout, o, a, grid, stream)
                      : launch_dq_layout<64, JATTN_SOFTMAX, true>(false, q, k, v, dout, o, a, grid, stream);
    return D == 128 ? launch_dq_layout<128, JATTN_SOFTMAX, false>(split, q, k, v, dout, o, a, grid, stream)
                    : launch_dq_layout<64, JATTN_SOFTMAX, false>(split, q, k, v, dout, o, a, grid, stream);
  }
#endif
  if (D == 128) {
    if (act == JATTN_SILU) return launch_dq_layout<128, JATTN_SILU, false>(split, q, k, v, dout, o, a, grid, stream);
    if (act == JATTN_GELU_POLY)
      return launch_dq_layout<128, JATTN_GELU_POLY, false>(split, q, k, v, dout, o, a, grid, stream);
    if (act == JATTN_GELU_TANH)
      return launch_dq_layout<128, JATTN_GELU_TANH, false>(split, q, k, v, dout, o, a, grid, stream);
    return cudaErrorInvalidValue;
  }
  if (act == JATTN_SILU) return launch_dq_layout<64, JATTN_SILU, false>(split, q, k, v, dout, o, a, grid, stream);
  if (act == JATTN_GELU_POLY)
    return launch_dq_layout<64, JATTN_GELU_POLY, false>(split, q, k, v, dout, o, a, grid, stream);
  if (act == JATTN_GELU_TANH)
    return launch_dq_layout<64, JATTN_GELU_TANH, false>(split, q, k, v, dout, o, a, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace jattn
