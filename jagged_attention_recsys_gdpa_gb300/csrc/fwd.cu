// Forward pass of jagged generalized dot-product attention on sm_103a.
//
// "GEM Training" post, section "Jagged Sequence Flash Attention" (FlashAttention
// run directly on the unpadded jagged tensors, warp specialisation, TMA and a
// persistent grid) and section "Generalized Dot-Product Attention" (the same
// two products with GELU/SiLU in place of softmax, which drops the online
// correction stage).
//
// One persistent CTA per SM walks the longest-first schedule. A work item is
// (sequence, 256-query block, head): two 128-row query tiles that share every
// K/V tile the producer streams in. Roles (12 warps, three warpgroups):
//   warp 0      TMA producer: Q tiles once per item, K and V tiles into two
//               rings (K one tile ahead of V)
//   warp 1      tcgen05 issuer: S_t = Q_t K_j^T into TMEM, O_t += P_t V_j
//               with P_t read straight from TMEM
//   warps 2-3   idle (their warpgroup gives its registers to the others)
//   warps 4-11  two activation warpgroups, in one of two arrangements:
//     ping-pong     warpgroup t owns query tile t: while one turns its S tile
//                   into P, the tensor core works on the other tile's products.
//                   P_t (bf16 pairs) overwrites S_t columns 0-63.
//     column split  both warpgroups work on every S tile, key columns 0-63 and
//                   64-127; P of each half overwrites the first 32 of the half's
//                   own S columns (0-31, 64-95), and softmax row maxima and sums
//                   are combined through shared memory. Items that hold a single
//                   query tile (short queries, e.g. pooling attention) keep all
//                   eight warps busy this way; the host picks the arrangement.
// TMEM columns: [S0 | S1 | O0 | O1].
// Softmax rescaling of O is lazy: the running maximum only moves (and O is
// rescaled in TMEM) when a row's maximum grows by more than 2^8.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

// This file is compiled four times: on its own for masks without the block
// bit, where the block-mask arithmetic folds away at compile time (left in, it
// cost the window-256 forward about 4%), through fwd_block.cu with
// JATTN_FWD_BLOCK = 1 for block masks, and through fwd_hilo.cu /
// fwd_block_hilo.cu with JATTN_HILO = 1 for pointwise activations without the
// 1/Lkv normaliser, whose P enters the PV product as bf16 hi + lo parts (the
// extra stores, even as branches not taken, slowed the normalised pooling
// forward by a quarter).
#ifndef JATTN_FWD_BLOCK
#define JATTN_FWD_BLOCK 0
#endif
#ifndef JATTN_HILO
#define JATTN_HILO 0
#endif

namespace jattn {

namespace {

constexpr int kNQ = 2;          // query tiles per item
constexpr int kThreads = 384;   // 12 warps: control warpgroup + two activation warpgroups
constexpr float kRescaleLog2 = 8.0f;
// Register split (setmaxnreg): 384 threads x 168 at launch = 64512 =
// 128 x 104 (control warpgroup) + 256 x 200 (activation warpgroups).
constexpr int kCtlRegs = 104;
constexpr int kActRegs = 200;

template <int D>
struct FwdCfg {
  static constexpr int kTileBytes = kTile * D * 2;   // one 128-row tile of Q, K or V
  static constexpr int kKStages = (D == 128) ? 3 : 6;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kNQ * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kXchOff = kBarOff + 512;                 // [2 slots][2 halves][128 rows] fp32
  static constexpr int kSmemBytes = kXchOff + 2 * 2 * kTile * 4;  // base is 1024-aligned (checked)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 2 * kTile;  // O_t at kOCol + t * D
};

struct FwdBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[6], k_empty[6], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t drain;
  uint64_t xbar[2][4];        // column split: row-exchange meeting per (slot, lane quarter), 64 arrivals
  uint32_t tmem_base;
  int abort_flag;
  volatile int okx[2][2][4];  // exchange slot, column half, lane quarter: partner still ok
};
static_assert(sizeof(FwdBars) <= 512, "barrier block overflows its slot");
static_assert(FwdCfg<128>::kSmemBytes <= 227 * 1024 && FwdCfg<64>::kSmemBytes <= 227 * 1024, "shared memory");

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// x * sigmoid(x) with sigmoid(x) = (1 + tanh(x/2)) / 2: one transcendental
// instead of an exponential and a reciprocal.
__device__ __forceinline__ float silu_f(float x) {
  const float h = 0.5f * x;
  return fmaf(h, tanh_approx(h), h);
}
__device__ __forceinline__ float gelu_f(float x) {
  const float u = 0.7978845608028654f * fmaf(0.044715f * x * x, x, x);
  return 0.5f * x * (1.0f + tanh_approx(u));
}
template <int ACT>
__device__ __forceinline__ float pointwise_f(float x) {
  if constexpr (ACT == JATTN_SILU) return silu_f(x);
  else if constexpr (ACT == JATTN_GELU_POLY) return gelu_poly(x);
  else return gelu_f(x);
}

// Wait bounded by time, ignoring the abort flag (teardown of in-flight copies).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

struct ItemInfo {
  int b, qb, lo, hi, h;
  int lq, lkv;
  int64_t q0, k0;
  int t_lo[kNQ], t_hi[kNQ];  // per query tile key-tile range (empty: lo == hi)
  bool t_rows[kNQ];          // tile has at least one query row
};

// The mask bits this compilation handles (see the top of the file).
__device__ __forceinline__ int kernel_mask(const AttnArgs& a) {
  return JATTN_FWD_BLOCK ? a.mask : (a.mask & ~JATTN_MASK_BLOCK);
}

__device__ __forceinline__ bool load_item(const AttnArgs& a, long long round, ItemInfo& it) {
  const long long n_items = static_cast<long long>(*a.n_tiles) * a.H;
  const long long k = zigzag_item(round, blockIdx.x, gridDim.x);
  if (k >= n_items) return false;
  const int4 t = a.tiles[k / a.H];
  it.h = static_cast<int>(k % a.H);
  it.b = t.x;
  it.qb = t.y;
  it.lo = t.z;
  it.hi = t.w;
  it.q0 = a.q_off[it.b];
  it.k0 = a.kv_off[it.b];
  it.lq = static_cast<int>(a.q_off[it.b + 1] - it.q0);
  it.lkv = static_cast<int>(a.kv_off[it.b + 1] - it.k0);
#pragma unroll
  for (int q = 0; q < kNQ; ++q) {
    const int rt = it.qb * kNQ + q;
    it.t_rows[q] = rt * kTile < it.lq;
    tile_range(it.lq, it.lkv, rt, kTile, kTile, kernel_mask(a), a.window, 0, it.t_lo[q], it.t_hi[q]);
  }
  return true;
}

template <int D, int ACT, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  using C = FwdCfg<D>;
  constexpr bool kHilo = JATTN_HILO && ACT != JATTN_SOFTMAX;  // P as bf16 hi + lo parts
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The tiles need 1024-byte alignment and the layout leaves no slack for
  // realigning, so a misaligned dynamic shared memory base is an error.
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(a.status, JATTN_ERR_UNSUPPORTED, 19, blockIdx.x);
    return;
  }
  uint8_t* sm = smem_raw;
  FwdBars* bars = reinterpret_cast<FwdBars*>(sm + C::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], (SPLIT ? 2 : 1) * kTile);
      mbar_init(&bars->o_full[t], 1);
      mbar_init(&bars->o_empty[t], (SPLIT ? 2 : 1) * kTile);
    }
    mbar_init(&bars->drain, 1);
    for (int x = 0; x < 2; ++x)
      for (int qq = 0; qq < 4; ++qq) mbar_init(&bars->xbar[x][qq], 64);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp < 4) {
  // The register split is set per warpgroup, at the same instruction for all
  // warps of the warpgroup, in the branch that holds the role's code.
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtlRegs));
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t k_it = 0, v_it = 0, q_it = 0;
      bool q_armed = false, ok = true;
      ItemInfo it;
      auto load_k = [&](int j) -> bool {
        const int s = k_it % C::kKStages;
        if (!wait_bar(&bars->k_empty[s], ((k_it / C::kKStages) & 1) ^ 1, abort_flag, a, 11)) return false;
        mbar_arrive_expect_tx(&bars->k_full[s], C::kTileBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sm + C::kKOff + s * C::kTileBytes + c * kTile * 128, &tmK, &bars->k_full[s],
                      it.h * D + c * 64, static_cast<int>(it.k0) + j * kTile);
        ++k_it;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = v_it % C::kVStages;
        if (!wait_bar(&bars->v_empty[s], ((v_it / C::kVStages) & 1) ^ 1, abort_flag, a, 12)) return false;
        mbar_arrive_expect_tx(&bars->v_full[s], C::kTileBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(sm + C::kVOff + s * C::kTileBytes + c * kTile * 128, &tmV, &bars->v_full[s],
                      it.h * D + c * 64, static_cast<int>(it.k0) + j * kTile);
        ++v_it;
        return true;
      };
      // the next item's descriptor is loaded while this one is served (its
      // global loads would otherwise stall every item start)
      ItemInfo nit;
      bool have = load_item(a, 0, it), have_next = false;
      for (long long r = 0; ok && have; ++r, it = nit, have = have_next) {
        have_next = load_item(a, r + 1, nit);
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->q_empty, (q_it & 1) ^ 1, abort_flag, a, 10))) break;
        if (!(a.debug_flags & 1)) {
          int nbytes = 0;
          for (int q = 0; q < kNQ; ++q) nbytes += it.t_rows[q] ? C::kTileBytes : 0;
          mbar_arrive_expect_tx(&bars->q_full, nbytes);
          for (int q = 0; q < kNQ; ++q) {
            if (!it.t_rows[q]) continue;
            const int y = static_cast<int>(it.q0) + (it.qb * kNQ + q) * kTile;
            for (int c = 0; c < D / 64; ++c)
              tma_load_2d(sm + C::kQOff + q * C::kTileBytes + c * kTile * 128, &tmQ, &bars->q_full,
                          it.h * D + c * 64, y);
          }
          q_armed = true;
        }
        ++q_it;
        // K runs one tile ahead of V: S(j+1) and P(j)V(j) are issued together.
        if (!(ok = load_k(it.lo))) break;
        for (int j = it.lo; j < it.hi && ok; ++j) {
          if (j + 1 < it.hi && !(ok = load_k(j + 1))) break;
          ok = load_v(j);
        }
      }
      // Let every copy this thread started land before the CTA can exit.
      if (q_armed) drain_wait(&bars->q_full, (q_it - 1) & 1, a.timeout_ns);
      for (uint32_t i = (k_it > (uint32_t)C::kKStages ? k_it - C::kKStages : 0); i < k_it; ++i)
        drain_wait(&bars->k_full[i % C::kKStages], (i / C::kKStages) & 1, a.timeout_ns);
      for (uint32_t i = (v_it > (uint32_t)C::kVStages ? v_it - C::kVStages : 0); i < v_it; ++i)
        drain_wait(&bars->v_full[i % C::kVStages], (i / C::kVStages) & 1, a.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kTile, kTile, false, false);
      constexpr uint32_t idPV = idesc_bf16_f32(kTile, D, false, true);
      const uint32_t sQ = smem_u32(sm + C::kQOff), sK = smem_u32(sm + C::kKOff), sV = smem_u32(sm + C::kVOff);
      uint32_t k_used = 0, v_used = 0, q_it = 0, p_cnt[2] = {0, 0}, o_cnt[2] = {0, 0};
      uint32_t k_waited = 0;  // 1 + index of the last K load whose barrier was waited
      bool ok = true;
      ItemInfo it;
      auto wait_k = [&](uint32_t idx) -> bool {
        if (k_waited == idx + 1) return true;
        if (!wait_bar(&bars->k_full[idx % C::kKStages], (idx / C::kKStages) & 1, abort_flag, a, 21)) return false;
        tc_fence_after();
        k_waited = idx + 1;
        return true;
      };
      // Shared-memory descriptors of the tile bases, computed once: the kk-th
      // 16-wide slice of a K-major tile lies (kk / 4) 64-column boxes and
      // (kk % 4) * 32 bytes further, and the next V slice 16 rows further,
      // which are additions to the descriptor's address field (16-byte units).
      // Each MMA then costs its issuing thread one add per operand.
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024), dK0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sV, kTile * 128, 1024);
      constexpr uint64_t kTileUnits = C::kTileBytes >> 4;
      auto kslice = [](int kk) -> uint64_t { return static_cast<uint64_t>(((kk >> 2) * (kTile * 128) + (kk & 3) * 32) >> 4); };
      auto issue_s = [&](int q, uint32_t kidx) {
        const uint64_t kd = dK0 + (kidx % C::kKStages) * kTileUnits, qd = dQ0 + q * kTileUnits;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tmem + q * kTile, qd + kslice(kk), kd + kslice(kk), idS, kk > 0);
        mma_commit(&bars->s_full[q]);
      };
      ItemInfo nit;
      bool have = load_item(a, 0, it), have_next = false;
      for (long long r = 0; ok && have; ++r, it = nit, have = have_next) {
        have_next = load_item(a, r + 1, nit);
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->q_full, q_it & 1, abort_flag, a, 20))) break;
        ++q_it;
        tc_fence_after();
        const uint32_t k0 = k_used, v0 = v_used;  // global load indices of this item's first K / V
        if (!(ok = wait_k(k0))) break;
#pragma unroll
        for (int q = 0; q < kNQ; ++q)
          if (it.t_lo[q] <= it.lo && it.lo < it.t_hi[q]) issue_s(q, k0);
        mma_commit(&bars->k_empty[k0 % C::kKStages]);
        // Q is free for the next item once the item's last S product completes.
        if (it.hi - it.lo == 1) mma_commit(&bars->q_empty);
        for (int j = it.lo; j < it.hi && ok; ++j) {
          const uint32_t vi = v0 + (j - it.lo), ki1 = k0 + (j - it.lo) + 1;
          const int vs = vi % C::kVStages;
          if (!(ok = wait_bar(&bars->v_full[vs], (vi / C::kVStages) & 1, abort_flag, a, 22))) break;
          tc_fence_after();
          if (j + 1 < it.hi && !(ok = wait_k(ki1))) break;
#pragma unroll
          for (int q = 0; q < kNQ; ++q) {
            if (!ok) break;
            if (it.t_lo[q] <= j && j < it.t_hi[q]) {
              if (j == it.t_lo[q]) {
                if (!(ok = wait_bar(&bars->o_empty[q], (o_cnt[q] & 1) ^ 1, abort_flag, a, 23))) break;
              }
              if (!(ok = wait_bar(&bars->p_full[q], p_cnt[q] & 1, abort_flag, a, 24))) break;
              ++p_cnt[q];
              tc_fence_after();
              const uint64_t vd = dV0 + vs * kTileUnits;
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk) {
                // P of key columns 16kk.. sits at column 8kk; with the column split,
                // at 8kk + 32 for the second half
                mma_ts(tmem + C::kOCol + q * D, tmem + q * kTile + kk * 8 + ((SPLIT && kk >= kTile / 32) ? 32 : 0),
                       vd + kk * (16 * 128 / 16), idPV, (kk > 0 || j > it.t_lo[q]) ? 1u : 0u);
              }
              if constexpr (kHilo) {
                // unnormalised pointwise: P's lo parts, 64 columns further (ping-pong)
                // or 32 further (column split); a rolled loop keeps the issuer's
                // registers within its share
#pragma unroll 1
                for (int kk = 0; kk < kTile / 16; ++kk)
                  mma_ts(tmem + C::kOCol + q * D,
                         tmem + q * kTile + kk * 8 + ((SPLIT && kk >= kTile / 32) ? 32 : 0) + (SPLIT ? 32 : 64),
                         vd + kk * (16 * 128 / 16), idPV, 1u);
              }
              if (j + 1 == it.t_hi[q]) {
                mma_commit(&bars->o_full[q]);
                ++o_cnt[q];
              }
            }
            if (j + 1 < it.hi && it.t_lo[q] <= j + 1 && j + 1 < it.t_hi[q]) issue_s(q, ki1);
          }
          if (!ok) break;
          if (j + 1 < it.hi) mma_commit(&bars->k_empty[ki1 % C::kKStages]);
          if (j + 2 == it.hi) mma_commit(&bars->q_empty);
          mma_commit(&bars->v_empty[vs]);
        }
        if (!ok) break;
        k_used += it.hi - it.lo;
        v_used += it.hi - it.lo;
      }
      // Every MMA this thread issued completes before TMEM is released.
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, a.timeout_ns);
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kActRegs));
    if constexpr (SPLIT) {
      // ------------------------------------------------------------ activation warpgroups
      // Both warpgroups work on every S tile, one column half each: warpgroup
      // `half` owns key columns [64 half, 64 half + 64) of S_t and O columns
      // [D/2 half, D/2 half + D/2) of O_t. Warp w and warp w ^ 4 hold the same
      // rows; for softmax they combine row maxima (every tile) and row sums
      // (epilogue) through shared memory.
      const int half = (warp - 4) >> 2;
      const int quarter = warp & 3;                   // TMEM lane quarter
      const int row = 32 * quarter + lane;            // TMEM lane == tile row
      const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
      constexpr int kHalfCols = kTile / 2;            // S columns of one half
      constexpr int kOHalf = D / 2;                   // O columns of one half
      float* xch = reinterpret_cast<float*>(sm + C::kXchOff);
      uint32_t s_cnt[kNQ] = {0, 0}, o_cnt[kNQ] = {0, 0}, x_cnt = 0;
      // Row exchange with the partner warp: both write their value and ok flag,
      // then meet on the (slot, quarter) mbarrier with a bounded wait, so a warp
      // whose partner has aborted gives up instead of waiting for it. Two slots,
      // alternating: a slot is rewritten only after the partner has arrived at
      // the meeting that follows its read.
      auto exchange = [&](float v, bool& okr) -> float {
        const int slot = x_cnt & 1;
        const uint32_t par = (x_cnt >> 1) & 1;
        ++x_cnt;
        xch[(slot * 2 + half) * kTile + row] = v;
        if (lane == 0) bars->okx[slot][half][quarter] = okr ? 1 : 0;
        mbar_arrive(&bars->xbar[slot][quarter]);
        const bool met = __all_sync(0xffffffffu, wait_bar(&bars->xbar[slot][quarter], par, abort_flag, a, 32));
        okr = okr && met && (bars->okx[slot][half ^ 1][quarter] != 0);
        return xch[(slot * 2 + (half ^ 1)) * kTile + row];
      };
      bool ok = true;
      ItemInfo it;
      for (long long r = 0; ok && load_item(a, r, it); ++r) {
        const int delta = it.lkv - it.lq;
        int klo[kNQ], khi[kNQ];
        float m_run[kNQ], l_run[kNQ];
#pragma unroll
        for (int q = 0; q < kNQ; ++q) {
          key_interval((it.qb * kNQ + q) * kTile + row, delta, it.lkv, kernel_mask(a), a.window, klo[q], khi[q]);
          if ((it.qb * kNQ + q) * kTile + row >= it.lq) khi[q] = klo[q];  // rows past the sequence see nothing
          m_run[q] = -INFINITY;
          l_run[q] = 0.0f;
        }
        for (int j = it.lo; ok && j < it.hi; ++j) {
#pragma unroll
          for (int q = 0; q < kNQ; ++q) {
            if (!ok) break;
            if (j < it.t_lo[q] || j >= it.t_hi[q]) continue;
            bool okw = wait_bar(&bars->s_full[q], s_cnt[q] & 1, abort_flag, a, 30);
            okw = __all_sync(0xffffffffu, okw);
            ++s_cnt[q];
            const uint32_t tS = tmem + lane_base + q * kTile + half * kHalfCols;
            float s[kHalfCols];
            if (okw) {
              tc_fence_after();
              uint32_t* su = reinterpret_cast<uint32_t*>(s);
              tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(su));
              tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(su + 32));
              tmem_ld_wait();
            }
            const int clo = klo[q] - j * kTile - half * kHalfCols, chi = khi[q] - j * kTile - half * kHalfCols;
            const bool edge = clo > 0 || chi < kHalfCols;
            // 32-column chunks that no row of this warp sees (rows past a short query
            // tile, masked corners) skip the arithmetic: their P is zero.
            bool skip[kHalfCols / 32];
#pragma unroll
            for (int k = 0; k < kHalfCols / 32; ++k) skip[k] = __all_sync(0xffffffffu, max(clo, 32 * k) >= min(chi, 32 * k + 32));
            if constexpr (ACT == JATTN_SOFTMAX) {
              float mx = -INFINITY;
              if (okw) {
                if (edge) {
#pragma unroll
                  for (int k = 0; k < kHalfCols / 32; ++k) {
                    if (skip[k]) continue;
#pragma unroll
                    for (int c = 32 * k; c < 32 * k + 32; ++c) s[c] = (c >= clo && c < chi) ? s[c] : -INFINITY;
                  }
                }
                // row maximum of this half: four independent chains of three-input maxima
                float mp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int k = 0; k < kHalfCols / 32; ++k) {
                  if (skip[k]) continue;
#pragma unroll
                  for (int c = 32 * k; c < 32 * k + 32; c += 8)
#pragma unroll
                    for (int e = 0; e < 4; ++e) mp[e] = fmax3(mp[e], s[c + 2 * e], s[c + 2 * e + 1]);
                }
                mx = fmax3(mp[0], mp[1], fmaxf(mp[2], mp[3]));
              }
              mx = fmaxf(mx, exchange(mx, okw));
              if (!okw) {
                ok = false;
                break;
              }
              const float m_new = mx * a.scale_log2;
              bool rescale = false;
              float alpha = 1.0f;
              if (m_run[q] == -INFINITY) {
                m_run[q] = m_new;  // O and l hold nothing yet for this row
              } else if (m_new > m_run[q] + kRescaleLog2) {
                alpha = ex2_approx(m_run[q] - m_new);
                rescale = true;
                m_run[q] = m_new;
                l_run[q] *= alpha;
              }
              if (__any_sync(0xffffffffu, rescale)) {
                // The previous P V product of this tile has completed: the S tile
                // just waited for was issued after it.
                const uint32_t tO = tmem + lane_base + C::kOCol + q * D + half * kOHalf;
#pragma unroll
                for (int c = 0; c < kOHalf / 16; ++c) {
                  uint32_t o[16];
                  tmem_ld16(tO + c * 16, o);
                  tmem_ld_wait();
#pragma unroll
                  for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                  tmem_st16(tO + c * 16, o);
                }
                tmem_st_wait();
              }
              const float mref = (m_run[q] == -INFINITY) ? 0.0f : m_run[q];
              // exponent arguments and row sums two lanes at a time (f32x2)
              const uint64_t c2 = f2(a.scale_log2, a.scale_log2), nm2 = f2(-mref, -mref);
              uint64_t ls2[4] = {0, 0, 0, 0};
#pragma unroll
              for (int c0 = 0; c0 < kHalfCols; c0 += 32) {
                uint32_t pk[16];
                if (skip[c0 / 32]) {
#pragma unroll
                  for (int e = 0; e < 16; ++e) pk[e] = 0u;
                  tmem_st16(tS + c0 / 2, pk);
                  continue;
                }
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                  float x0, x1;
                  f2_split(ffma2(f2(s[c0 + e], s[c0 + e + 1]), c2, nm2), x0, x1);
                  const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                  ls2[(e >> 1) & 3] = fadd2(ls2[(e >> 1) & 3], f2(p0, p1));
                  pk[e / 2] = pack_bf16x2(p0, p1);
                }
                // P of this half goes to the first 32 columns of the half's own S
                // columns, which this warp has already read
                tmem_st16(tS + c0 / 2, pk);
              }
              float l0, l1;
              f2_split(fadd2(fadd2(ls2[0], ls2[1]), fadd2(ls2[2], ls2[3])), l0, l1);
              l_run[q] += l0 + l1;
            } else {
              if (!okw) {
                ok = false;
                break;
              }
#pragma unroll
              for (int c0 = 0; c0 < kHalfCols; c0 += 32) {
                uint32_t pk[16];
                if (skip[c0 / 32]) {
#pragma unroll
                  for (int e = 0; e < 16; ++e) pk[e] = 0u;
                  tmem_st16(tS + c0 / 2, pk);
                  if constexpr (kHilo) tmem_st16(tS + 32 + c0 / 2, pk);
                  continue;
                }
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                  const int c = c0 + e;
                  const float x0 = s[c] * a.scale, x1 = s[c + 1] * a.scale;
                  float p0 = pointwise_f<ACT>(x0);
                  float p1 = pointwise_f<ACT>(x1);
                  if (edge) {
                    p0 = (c >= clo && c < chi) ? p0 : 0.0f;
                    p1 = (c + 1 >= clo && c + 1 < chi) ? p1 : 0.0f;
                  }
                  pk[e / 2] = pack_bf16x2(p0, p1);
                  // lo parts (unnormalised mode) in the half's other 32 columns, already read
                  if constexpr (kHilo) tmem_st1(tS + 32 + (c0 + e) / 2, bf16x2_lo(p0, p1, pk[e / 2]));
                }
                tmem_st16(tS + c0 / 2, pk);
              }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars->p_full[q]);
          }
        }
        if (!ok) break;
        // ---------------- epilogue: each half stores its O columns of each tile
#pragma unroll
        for (int q = 0; q < kNQ; ++q) {
          if (!ok) break;
          if (!it.t_rows[q]) continue;
          const int row_local = (it.qb * kNQ + q) * kTile + row;
          const bool valid = row_local < it.lq;
          const int64_t grow = it.q0 + row_local;
          const int n = (it.hi > it.lo) ? (it.t_hi[q] - it.t_lo[q]) : 0;
          bool okw = true;
          if (n > 0) {
            okw = wait_bar(&bars->o_full[q], o_cnt[q] & 1, abort_flag, a, 31);
            okw = __all_sync(0xffffffffu, okw);
            ++o_cnt[q];
          }
          float l_tot = l_run[q];
          if constexpr (ACT == JATTN_SOFTMAX) l_tot += exchange(l_run[q], okw);
          if (!okw) {
            ok = false;
            break;
          }
          float oscale;
          if constexpr (ACT == JATTN_SOFTMAX) {
            oscale = (l_tot > 0.0f) ? 1.0f / l_tot : 0.0f;
          } else {
            oscale = (a.norm_by_lkv && it.lkv > 0) ? 1.0f / static_cast<float>(it.lkv) : 1.0f;
          }
          __nv_bfloat16* orow = a.out0 + (grow * a.H + it.h) * D + half * kOHalf;
          if (n > 0) {
            tc_fence_after();
            const uint32_t tO = tmem + lane_base + C::kOCol + q * D + half * kOHalf;
#pragma unroll
            for (int c = 0; c < kOHalf / 32; ++c) {
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
            mbar_arrive(&bars->o_empty[q]);
          } else if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow);
            for (int e = 0; e < kOHalf / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
          }
          if constexpr (ACT == JATTN_SOFTMAX) {
            if (valid && half == 0 && a.f0 != nullptr) {  // block masks may leave LSE out
              const float lse = (l_tot > 0.0f) ? (m_run[q] + __log2f(l_tot)) * 0.6931471805599453f : -INFINITY;
              a.f0[grow * a.H + it.h] = lse;
            }
          }
        }
      }
    } else {
      // Ping-pong: warpgroup q owns query tile q of the item; while one turns
      // its S tile into P, the tensor core works on the other tile.
      // ------------------------------------------------------------ activation warpgroups
      const int q = (warp - 4) >> 2;                 // query tile of this warpgroup
      const int row = 32 * (warp & 3) + lane;         // TMEM lane == tile row
      const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
      const uint32_t tS = tmem + lane_base + q * kTile;
      const uint32_t tO = tmem + lane_base + C::kOCol + q * D;
      uint32_t s_cnt = 0, o_cnt = 0;
      ItemInfo it;
      for (long long r = 0; load_item(a, r, it); ++r) {
        const bool has_rows = q ? it.t_rows[1] : it.t_rows[0];
        const int t_lo = q ? it.t_lo[1] : it.t_lo[0];
        const int t_hi = q ? it.t_hi[1] : it.t_hi[0];
        if (!has_rows) continue;
        const int row_local = (it.qb * kNQ + q) * kTile + row;
        const bool valid = row_local < it.lq;
        const int64_t grow = it.q0 + row_local;
        const int delta = it.lkv - it.lq;
        int klo, khi;
        key_interval(row_local, delta, it.lkv, kernel_mask(a), a.window, klo, khi);
        const int n = (it.hi > it.lo) ? (t_hi - t_lo) : 0;
        float m_run = -INFINITY, l_run = 0.0f;
        bool ok = true;
        for (int j = t_lo; j < t_lo + n; ++j) {
          ok = wait_bar(&bars->s_full[q], s_cnt & 1, abort_flag, a, 30);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          ++s_cnt;
          tc_fence_after();
          float s[kTile];
          {
            uint32_t* su = reinterpret_cast<uint32_t*>(s);
#pragma unroll
            for (int c = 0; c < kTile / 32; ++c)
              tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(su + c * 32));
            tmem_ld_wait();
          }
          const int clo = klo - j * kTile, chi = khi - j * kTile;
          const bool edge = clo > 0 || chi < kTile;
          if constexpr (ACT == JATTN_SOFTMAX) {
            if (edge) {
#pragma unroll
              for (int c = 0; c < kTile; ++c) s[c] = (c >= clo && c < chi) ? s[c] : -INFINITY;
            }
            // row maximum: four independent chains of three-input maxima
            float mp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < kTile; c += 8)
#pragma unroll
              for (int e = 0; e < 4; ++e) mp[e] = fmax3(mp[e], s[c + 2 * e], s[c + 2 * e + 1]);
            const float mx = fmax3(mp[0], mp[1], fmaxf(mp[2], mp[3]));
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
              // The previous P V product of this tile has completed: the S tile
              // just waited for was issued after it.
#pragma unroll
              for (int c = 0; c < D / 16; ++c) {
                uint32_t o[16];
                tmem_ld16(tO + c * 16, o);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st16(tO + c * 16, o);
              }
              tmem_st_wait();
            }
            const float mref = (m_run == -INFINITY) ? 0.0f : m_run;
            // exponent arguments and row sums two lanes at a time (f32x2)
            const uint64_t c2 = f2(a.scale_log2, a.scale_log2), nm2 = f2(-mref, -mref);
            uint64_t ls2[4] = {0, 0, 0, 0};
#pragma unroll
            for (int c0 = 0; c0 < kTile; c0 += 32) {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float x0, x1;
                f2_split(ffma2(f2(s[c0 + e], s[c0 + e + 1]), c2, nm2), x0, x1);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                ls2[(e >> 1) & 3] = fadd2(ls2[(e >> 1) & 3], f2(p0, p1));
                pk[e / 2] = pack_bf16x2(p0, p1);
              }
              // P columns [c0/2, c0/2+16) only overlap S columns already read
              tmem_st16(tS + c0 / 2, pk);
            }
            float l0, l1;
            f2_split(fadd2(fadd2(ls2[0], ls2[1]), fadd2(ls2[2], ls2[3])), l0, l1);
            l_run += l0 + l1;
          } else {
#pragma unroll
            for (int c0 = 0; c0 < kTile; c0 += 32) {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                const int c = c0 + e;
                const float x0 = s[c] * a.scale, x1 = s[c + 1] * a.scale;
                float p0 = pointwise_f<ACT>(x0);
                float p1 = pointwise_f<ACT>(x1);
                if (edge) {
                  p0 = (c >= clo && c < chi) ? p0 : 0.0f;
                  p1 = (c + 1 >= clo && c + 1 < chi) ? p1 : 0.0f;
                }
                pk[e / 2] = pack_bf16x2(p0, p1);
                // lo parts (unnormalised mode) in columns 64.., whose scores are in registers
                if constexpr (kHilo) tmem_st1(tS + 64 + (c0 + e) / 2, bf16x2_lo(p0, p1, pk[e / 2]));
              }
              tmem_st16(tS + c0 / 2, pk);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->p_full[q]);
        }
        if (!ok) break;
        // ---------------- epilogue
        float oscale;
        if constexpr (ACT == JATTN_SOFTMAX) {
          oscale = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
        } else {
          oscale = (a.norm_by_lkv && it.lkv > 0) ? 1.0f / static_cast<float>(it.lkv) : 1.0f;
        }
        __nv_bfloat16* orow = a.out0 + (grow * a.H + it.h) * D;
        if (n > 0) {
          ok = wait_bar(&bars->o_full[q], o_cnt & 1, abort_flag, a, 31);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          ++o_cnt;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
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
          mbar_arrive(&bars->o_empty[q]);
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
          for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
        }
        if constexpr (ACT == JATTN_SOFTMAX) {
          if (valid && a.f0 != nullptr) {  // block masks may leave LSE out
            const float lse = (l_run > 0.0f) ? (m_run + __log2f(l_run)) * 0.6931471805599453f : -INFINITY;
            a.f0[grow * a.H + it.h] = lse;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

}  // namespace

template <int D, int ACT, bool SPLIT>
static cudaError_t launch_fwd_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const AttnArgs& a, int grid, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kern = fwd_kernel<D, ACT, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(q, k, v, a);
  return cudaGetLastError();
}

template <int D, int ACT>
static cudaError_t launch_fwd_s(bool split, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const AttnArgs& a, int grid, cudaStream_t stream) {
  return split ? launch_fwd_t<D, ACT, true>(q, k, v, a, grid, stream)
               : launch_fwd_t<D, ACT, false>(q, k, v, a, grid, stream);
}

#if JATTN_FWD_BLOCK && JATTN_HILO
cudaError_t launch_fwd_block_hilo(int D, int act, bool split, const CUtensorMap& q, const CUtensorMap& k,
                                  const CUtensorMap& v, const AttnArgs& a, int grid, cudaStream_t stream) {
#elif JATTN_FWD_BLOCK
cudaError_t launch_fwd_block(int D, int act, bool split, const CUtensorMap& q, const CUtensorMap& k,
                             const CUtensorMap& v, const AttnArgs& a, int grid, cudaStream_t stream) {
#elif JATTN_HILO
cudaError_t launch_fwd_hilo(int D, int act, bool split, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, const AttnArgs& a, int grid, cudaStream_t stream) {
#else
cudaError_t launch_fwd(int D, int act, bool split, bool block, bool hilo, const CUtensorMap& q, const CUtensorMap& k,
                       const CUtensorMap& v, const AttnArgs& a, int grid, cudaStream_t stream) {
  if (hilo && act != JATTN_SOFTMAX)
    return block ? launch_fwd_block_hilo(D, act, split, q, k, v, a, grid, stream)
                 : launch_fwd_hilo(D, act, split, q, k, v, a, grid, stream);
  if (block) return launch_fwd_block(D, act, split, q, k, v, a, grid, stream);
#endif
#if !JATTN_HILO
  if (D == 128 && act == JATTN_SOFTMAX) return launch_fwd_s<128, JATTN_SOFTMAX>(split, q, k, v, a, grid, stream);
  if (D == 64 && act == JATTN_SOFTMAX) return launch_fwd_s<64, JATTN_SOFTMAX>(split, q, k, v, a, grid, stream);
#endif
  if (D == 128) {
    if (act == JATTN_SILU) return launch_fwd_s<128, JATTN_SILU>(split, q, k, v, a, grid, stream);
    if (act == JATTN_GELU_POLY) return launch_fwd_s<128, JATTN_GELU_POLY>(split, q, k, v, a, grid, stream);
    if (act == JATTN_GELU_TANH) return launch_fwd_s<128, JATTN_GELU_TANH>(split, q, k, v, a, grid, stream);
    return cudaErrorInvalidValue;
  }
  if (act == JATTN_SILU) return launch_fwd_s<64, JATTN_SILU>(split, q, k, v, a, grid, stream);
  if (act == JATTN_GELU_POLY) return launch_fwd_s<64, JATTN_GELU_POLY>(split, q, k, v, a, grid, stream);
  if (act == JATTN_GELU_TANH) return launch_fwd_s<64, JATTN_GELU_TANH>(split, q, k, v, a, grid, stream);
  return cudaErrorInvalidValue;
}

#if !JATTN_FWD_BLOCK && !JATTN_HILO
int fwd_rows_per_item() { return kNQ * kTile; }
#endif

}  // namespace jattn
