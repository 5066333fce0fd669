// Attention with the keys on the MMA's M dimension, for sequences that are
// short on one side, on sm_103a.
//
// "GEM Training" post, section "Generalized Dot-Product Attention (GDPA)":
// pooling attention (PMA) runs a few learned queries per sequence against the
// sequence's keys with a pointwise activation, and cross-attention often sees
// short K/V. A 128-row query tile holding 32 queries leaves three quarters of
// every MMA's M rows empty. Here the products are transposed so that 128 keys
// fill M and at most 64 queries are the N dimension:
//   forward   S^T = K Q^T; P^T = act(scale S^T) goes to shared memory as
//             bf16; O^T += V^T P^T (M = head dim) accumulates in TMEM over the
//             key tiles, and O is written from O^T at the item's end. Items
//             are 64-query pieces from the 64-row query-tile schedule.
//   backward  one item = (sequence, head); each step computes S^T = K Q^T and
//             dP^T = V dO^T, P^T and dS^T = act'(scale S^T) * dP^T, then
//             dV += P^T dO, dK += dS^T Q and dQ^T += K^T dS^T, with all five
//             products once (none recomputed). Two modes:
//     pooling   (every sequence 1 <= Lq <= 64, or no keys): the queries are
//               loaded once, the key tiles are the steps; dV and dK of a tile
//               are complete after its step, dQ^T accumulates over the item.
//               K and V are read once and dK / dV written once: there is no
//               second pass that reads K and V again for dQ.
//     cross     (every sequence Lkv <= 128, and keys when it has queries): the
//               K / V tile is loaded once, the 64-query chunks are the steps;
//               dQ of a chunk is complete after its step, dV and dK
//               accumulate over the item. Q and dO are read once. Only
//               behind debug flag bit 128: the short-key backward below
//               takes these shapes.
// The same short-key shapes run in the usual orientation (queries on N):
// skv_fwd_kernel keeps each sequence's K / V tile in shared memory while its
// 128-row query tiles stream through a ring, and skv_bwd_kernel does the same
// for the backward, with 128 queries per step so that all five products run
// at N = 128.
// A gate kernel checks the chosen mode's limits on the device and either
// clears the general dQ and dK/dV schedules (their passes then find no work)
// or leaves them to run while this pass finds the gate closed and returns.
//
// Roles: warp 0 issues TMA copies, warp 1 issues tcgen05 MMAs. The forward's
// two activation warpgroups (warps 4-7, 8-11) take alternate key tiles; the
// backward's (same warps) split every step's 64 query columns, and an
// epilogue warpgroup (warps 12-15) drains dV / dK and dQ. Thread i of a
// warpgroup owns TMEM lane i: a key row of S^T / dP^T / dV / dK, or a
// head-dim row of O^T / dQ^T.
//
// Pointwise activations without the 1/Lkv normaliser pass P and dS to the
// second products as bf16 hi + lo parts (template HILO), as the general
// kernels do: outputs there sum thousands of unscaled terms.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace jattn {

namespace {

constexpr int kD = 128;                      // head dim (the only one this path takes)
constexpr int kQC = 64;                      // query rows of an item: the MMAs' N
constexpr int kThreads = 384;                // 12 warps
constexpr int kBoxK = kTile * 128;           // one [128 rows][64 columns] bf16 box (16 KB)
constexpr int kBoxQ = kQC * 128;             // one [64 rows][64 columns] bf16 box (8 KB)
constexpr int kTileBytes = 2 * kBoxK;        // K or V tile: [128 keys][128]
constexpr int kChunkBytes = 2 * kBoxQ;       // Q or dO chunk: [64 queries][128]
constexpr int kPBytes = kTile * kQC * 2;     // P^T or dS^T: [128 keys][64 queries] bf16
constexpr float kLog2e = 1.4426950408889634f;
// Backward: 16 warps, register split (setmaxnreg, per warpgroup): 512 x 128
// at launch = 65536 >= 128 x (control + 2 activation + epilogue). Each
// activation thread holds a key row's 32 scores and 32 activation
// derivatives. A warpgroup that ends below the launch count lowers its share
// (.dec), one above it raises it (.inc): .inc may not ask for fewer registers
// than the warp holds.
constexpr int kBwdThreads = 512;
constexpr int kLaunchRegs = 128;
constexpr int kCtlRegs = 136;
constexpr int kActRegs = 128;
constexpr int kEpiRegs = 120;
static_assert(128 * (kCtlRegs + 2 * kActRegs + kEpiRegs) <= kBwdThreads * kLaunchRegs, "register split");
static_assert(kCtlRegs >= kLaunchRegs && kEpiRegs <= kLaunchRegs && kActRegs == kLaunchRegs,
              "dec / inc directions of the split");

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// act(x) and act'(x) of the pointwise activations (SiLU, tanh-GELU, and
// tanh-GELU's Taylor polynomial).
template <int ACT>
__device__ __forceinline__ void act_and_grad(float x, float& f, float& g) {
  if constexpr (ACT == JATTN_SILU) {
    // with h = x / 2 and t = tanh h: sigmoid(x) = (1 + t) / 2, so
    // f = h (1 + t) and f' = (1 + t + h (1 - t^2)) / 2 (one MUFU operation)
    const float h = 0.5f * x;
    const float t = tanh_approx(h);
    f = fmaf(h, t, h);
    g = fmaf(0.5f, t + fmaf(-h, t * t, h), 0.5f);
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
template <int ACT>
__device__ __forceinline__ float act_f(float x) {
  if constexpr (ACT == JATTN_SILU) {
    const float h = 0.5f * x;  // x sigmoid(x) = h (1 + tanh h)
    return fmaf(h, tanh_approx(h), h);
  } else if constexpr (ACT == JATTN_GELU_POLY) {
    return gelu_poly(x);
  } else {
    const float u = 0.7978845608028654f * fmaf(0.044715f * x * x, x, x);
    return 0.5f * x * (1.0f + tanh_approx(u));
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// 16 packed bf16 pairs (queries c0 .. c0 + 31 of key row `row`) into a
// [128 keys][64 queries] tile in the 128-byte-swizzled layout an MN-major MMA
// operand reads: row r at r * 128 bytes, its 16-byte piece p at (p ^ (r & 7)).
__device__ __forceinline__ void st_pt_row(uint32_t tile, int row, int c0, const uint32_t (&w)[16]) {
  const uint32_t base = tile + static_cast<uint32_t>(row) * 128;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int piece = (c0 >> 3) + i;
    st_shared_v4(base + ((piece ^ (row & 7)) << 4), w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return;
  }
}

// Descriptor offsets (16-byte units). K-major operands: the kk-th 16-wide
// slice of a 128-column row lies (kk / 4) boxes and (kk % 4) * 32 bytes
// further. MN-major operands: the kk-th 16-row slice lies 16 rows further.
__device__ __forceinline__ uint64_t kslice(int kk, int box_bytes) {
  return static_cast<uint64_t>(((kk >> 2) * box_bytes + (kk & 3) * 32) >> 4);
}
__device__ __forceinline__ uint64_t mnslice(int kk) { return static_cast<uint64_t>((kk * 16 * 128) >> 4); }

struct PItem {
  int b, rt, lo, hi, h, lq, lkv;  // lq: query rows of this item (at most kQC)
  int64_t q0, k0;                 // first query row of the item, first key row of the sequence
};

__device__ __forceinline__ bool load_pitem(const AttnArgs& a, long long round, PItem& it) {
  const long long n_items = static_cast<long long>(*a.n_tiles) * a.H;
  const long long k = zigzag_item(round, blockIdx.x, gridDim.x);
  if (k >= n_items) return false;
  const int4 t = a.tiles[k / a.H];
  it.h = static_cast<int>(k % a.H);
  it.b = t.x;
  it.rt = t.y;
  it.lo = t.z;
  it.hi = t.w;
  const int64_t qs = a.q_off[it.b];
  it.q0 = qs + static_cast<int64_t>(it.rt) * kQC;
  const int64_t rest = a.q_off[it.b + 1] - it.q0;
  it.lq = static_cast<int>(rest < kQC ? rest : kQC);
  it.k0 = a.kv_off[it.b];
  it.lkv = static_cast<int>(a.kv_off[it.b + 1] - it.k0);
  return true;
}

// One output element per (query, head-dim row): thread d of a warpgroup
// writes O[q][h][d] (or dQ) for the queries [c0, c0 + 32) below lq, from 32
// fp32 accumulator columns (nullptr: zeros). A warp's 32 lanes write 64
// contiguous bytes per query.
__device__ __forceinline__ void store_cols(__nv_bfloat16* out, const PItem& it, int H, int d, int c0,
                                           const uint32_t* v, float mul) {
  for (int e = 0; e < 32; ++e) {
    const int q = c0 + e;
    if (q >= it.lq) break;
    const float x = v ? __uint_as_float(v[e]) * mul : 0.0f;
    out[((it.q0 + q) * H + it.h) * kD + d] = __float2bfloat16_rn(x);
  }
}

// ---------------------------------------------------------------------------- forward
template <bool HILO>
struct PfCfg {
  static constexpr int kKStages = HILO ? 2 : 3;
  static constexpr int kVStages = 2;
  static constexpr int kNP = HILO ? 2 : 1;  // P^T tiles per buffer (hi, lo)
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kChunkBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kPOff = kVOff + kVStages * kTileBytes;  // [2 buffers][kNP] P^T tiles
  static constexpr int kBarOff = kPOff + 2 * kNP * kPBytes;
  static constexpr int kSmemBytes = kBarOff + 256;
  static constexpr uint32_t kOCol = 2 * kQC;  // S^T buffers at 0 and 64, O^T after them
};
static_assert(PfCfg<false>::kSmemBytes <= 227 * 1024 && PfCfg<true>::kSmemBytes <= 227 * 1024, "shared memory");

struct PfBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full[2], s_free[2], p_full[2], p_free[2];
  uint64_t o_full, o_empty, drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(PfBars) <= 256, "barrier block overflows its slot");

template <int ACT, bool HILO>
__global__ void __launch_bounds__(kThreads, 1)
    pma_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  using C = PfCfg<HILO>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(a.status, JATTN_ERR_UNSUPPORTED, 80, blockIdx.x);
    return;
  }
  uint8_t* sm = smem_raw;
  PfBars* bars = reinterpret_cast<PfBars*>(sm + C::kBarOff);
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
    for (int g = 0; g < 2; ++g) {
      mbar_init(&bars->s_full[g], 1);
      mbar_init(&bars->s_free[g], kTile);
      mbar_init(&bars->p_full[g], kTile);
      mbar_init(&bars->p_free[g], 1);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 2 * kTile);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 256);
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
      uint32_t k_it = 0, v_it = 0, q_it = 0;
      bool q_armed = false, ok = true;
      PItem it;
      auto load_kv = [&](const CUtensorMap* map, uint64_t* full, uint64_t* empty, int stages, int off, uint32_t& cnt,
                         int j, int where) -> bool {
        const int s = cnt % stages;
        if (!wait_bar(&empty[s], ((cnt / stages) & 1) ^ 1, abort_flag, a, where)) return false;
        mbar_arrive_expect_tx(&full[s], kTileBytes);
        for (int c = 0; c < 2; ++c)
          tma_load_2d(sm + off + s * kTileBytes + c * kBoxK, map, &full[s], it.h * kD + c * 64,
                      static_cast<int>(it.k0) + j * kTile);
        ++cnt;
        return true;
      };
      for (long long r = 0; ok && load_pitem(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->q_empty, (q_it & 1) ^ 1, abort_flag, a, 81))) break;
        if (!(a.debug_flags & 1)) {
          mbar_arrive_expect_tx(&bars->q_full, kChunkBytes);
          for (int c = 0; c < 2; ++c)
            tma_load_2d(sm + C::kQOff + c * kBoxQ, &tmQ, &bars->q_full, it.h * kD + c * 64, static_cast<int>(it.q0));
          q_armed = true;
        }
        ++q_it;
        // K runs a tile ahead of V: S^T(j + 1) is issued before O^T's product with P^T(j).
        if (!(ok = load_kv(&tmK, bars->k_full, bars->k_empty, C::kKStages, C::kKOff, k_it, it.lo, 82))) break;
        for (int j = it.lo; j < it.hi && ok; ++j) {
          if (j + 1 < it.hi && !(ok = load_kv(&tmK, bars->k_full, bars->k_empty, C::kKStages, C::kKOff, k_it, j + 1, 82)))
            break;
          ok = load_kv(&tmV, bars->v_full, bars->v_empty, C::kVStages, C::kVOff, v_it, j, 83);
        }
      }
      // every copy this thread started lands before the CTA can exit
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
      constexpr uint32_t idS = idesc_bf16_f32(kTile, kQC, false, false);  // S^T = K Q^T
      constexpr uint32_t idO = idesc_bf16_f32(kD, kQC, true, true);       // O^T += V^T P^T
      const uint32_t sQ = smem_u32(sm + C::kQOff), sK = smem_u32(sm + C::kKOff), sV = smem_u32(sm + C::kVOff);
      const uint32_t sP = smem_u32(sm + C::kPOff);
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024), dK0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t dVt0 = sdesc_sw128(sV, kBoxK, 1024), dP0 = sdesc_sw128(sP, kPBytes, 1024);
      uint32_t k_used = 0, v_used = 0, q_it = 0, o_cnt = 0, n = 0;
      bool ok = true;
      PItem it;
      // O^T += V^T P^T of the item's t-th key tile (global tile index nt)
      auto issue_o = [&](int t, uint32_t nt) -> bool {
        const uint32_t vi = v_used + t, g = nt & 1, u = nt >> 1;
        const int vs = vi % C::kVStages;
        if (!wait_bar(&bars->v_full[vs], (vi / C::kVStages) & 1, abort_flag, a, 84)) return false;
        if (!wait_bar(&bars->p_full[g], u & 1, abort_flag, a, 85)) return false;
        if (t == 0 && !wait_bar(&bars->o_empty, (o_cnt & 1) ^ 1, abort_flag, a, 86)) return false;
        tc_fence_after();
        const uint64_t vd = dVt0 + vs * (kTileBytes >> 4);
#pragma unroll
        for (int hl = 0; hl < C::kNP; ++hl) {
          const uint64_t pd = dP0 + (g * C::kNP + hl) * (kPBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ss(tmem + C::kOCol, vd + mnslice(kk), pd + mnslice(kk), idO, (t > 0 || hl > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars->p_free[g]);
        mma_commit(&bars->v_empty[vs]);
        return true;
      };
      for (long long r = 0; ok && load_pitem(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->q_full, q_it & 1, abort_flag, a, 87))) break;
        ++q_it;
        tc_fence_after();
        const int nk = it.hi - it.lo;
        for (int t = 0; t < nk && ok; ++t) {
          const uint32_t ki = k_used + t, nt = n + t, g = nt & 1, u = nt >> 1;
          const int ks = ki % C::kKStages;
          if (!(ok = wait_bar(&bars->k_full[ks], (ki / C::kKStages) & 1, abort_flag, a, 88))) break;
          if (!(ok = wait_bar(&bars->s_free[g], (u & 1) ^ 1, abort_flag, a, 89))) break;
          tc_fence_after();
          const uint64_t kd = dK0 + ks * (kTileBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_ss(tmem + g * kQC, kd + kslice(kk, kBoxK), dQ + kslice(kk, kBoxQ), idS, kk > 0 ? 1u : 0u);
          mma_commit(&bars->s_full[g]);
          mma_commit(&bars->k_empty[ks]);
          if (t == nk - 1) mma_commit(&bars->q_empty);  // Q is read by the S^T products only
          if (t > 0) ok = issue_o(t - 1, nt - 1);
        }
        if (ok) ok = issue_o(nk - 1, n + nk - 1);
        if (!ok) break;
        mma_commit(&bars->o_full);
        ++o_cnt;
        n += nk;
        k_used += nk;
        v_used += nk;
      }
      // every MMA this thread issued completes before TMEM is released
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, a.timeout_ns);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ activation warpgroups
    // Warpgroup g takes the key tiles of odd / even global index: S^T buffer
    // g in TMEM, P^T buffer g in shared memory. At an item's end both read
    // O^T, queries [32 g, 32 g + 32) each.
    const int g = (warp - 4) >> 2;
    const int row = 32 * (warp & 3) + lane;  // key row of S^T; head-dim row of O^T
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t sP = smem_u32(sm + C::kPOff);
    uint32_t n = 0, o_cnt = 0;
    bool ok = true;
    PItem it;
    for (long long r = 0; ok && load_pitem(a, r, it); ++r) {
      __nv_bfloat16* out = a.out0;
      if (it.hi <= it.lo) {  // no keys: the item's output rows are zero
        store_cols(out, it, a.H, row, 32 * g, nullptr, 0.0f);
        continue;
      }
      const int nk = it.hi - it.lo;
      for (int t = 0; t < nk; ++t) {
        const uint32_t nt = n + t;
        if ((nt & 1) != static_cast<uint32_t>(g)) continue;
        const uint32_t u = nt >> 1;
        ok = __all_sync(0xffffffffu, wait_bar(&bars->s_full[g], u & 1, abort_flag, a, 90));
        if (!ok) break;
        tc_fence_after();
        uint32_t s[kQC];
#pragma unroll
        for (int c = 0; c < kQC / 32; ++c)
          if (32 * c < it.lq) tmem_ld32(tmem + lane_base + g * kQC + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(s + 32 * c));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bars->s_free[g]);
        // keys past the sequence (a ragged last tile) give P = 0; columns past
        // the item's queries only reach O^T columns that are never stored
        const bool valid = (it.lo + t) * kTile + row < it.lkv;
        ok = __all_sync(0xffffffffu, wait_bar(&bars->p_free[g], (u & 1) ^ 1, abort_flag, a, 91));
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < kQC / 32; ++c) {
          if (32 * c >= it.lq) continue;
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float f0 = valid ? act_f<ACT>(__uint_as_float(s[32 * c + 2 * e]) * a.scale) : 0.0f;
            const float f1 = valid ? act_f<ACT>(__uint_as_float(s[32 * c + 2 * e + 1]) * a.scale) : 0.0f;
            hi[e] = pack_bf16x2(f0, f1);
            if constexpr (HILO) lo[e] = bf16x2_lo(f0, f1, hi[e]);
          }
          st_pt_row(sP + (g * C::kNP) * kPBytes, row, 32 * c, hi);
          if constexpr (HILO) st_pt_row(sP + (g * C::kNP + 1) * kPBytes, row, 32 * c, lo);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->p_full[g]);
      }
      if (!ok) break;
      n += nk;
      // epilogue: O^T columns [32 g, 32 g + 32), times 1/Lkv when asked
      ok = __all_sync(0xffffffffu, wait_bar(&bars->o_full, o_cnt & 1, abort_flag, a, 92));
      if (!ok) break;
      ++o_cnt;
      tc_fence_after();
      const float cn = (a.norm_by_lkv && it.lkv > 0) ? 1.0f / it.lkv : 1.0f;
      uint32_t v[32];
      if (32 * g < it.lq) {
        tmem_ld32(tmem + lane_base + C::kOCol + 32 * g, v);
        tmem_ld_wait();
      }
      tc_fence_before();
      mbar_arrive(&bars->o_empty);
      if (32 * g < it.lq) store_cols(out, it, a.H, row, 32 * g, v, cn);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// Item of the fused backward: pooling items come from the 64-row query-tile
// schedule (one tile per sequence; [lo, hi) = key tiles), cross items from
// the 128-row key-tile schedule with 64-column query ranges (one tile per
// sequence; [lo, hi) = query chunks).
template <bool CROSS>
__device__ __forceinline__ bool load_bitem(const AttnArgs& a, long long round, PItem& it) {
  if constexpr (!CROSS) {
    return load_pitem(a, round, it);
  } else {
    const long long n_items = static_cast<long long>(*a.n_tiles) * a.H;
    const long long k = zigzag_item(round, blockIdx.x, gridDim.x);
    if (k >= n_items) return false;
    const int4 t = a.tiles[k / a.H];
    it.h = static_cast<int>(k % a.H);
    it.b = t.x;
    it.rt = t.y;  // key tile (0: the gate admits at most 128 keys)
    it.lo = t.z;
    it.hi = t.w;
    it.q0 = a.q_off[it.b];
    it.lq = static_cast<int>(a.q_off[it.b + 1] - it.q0);
    it.k0 = a.kv_off[it.b];
    it.lkv = static_cast<int>(a.kv_off[it.b + 1] - it.k0);
    return true;
  }
}

// Queries [c0, c0 + 32) of a chunk whose first row is q_first and which holds
// nq rows: thread d writes out[q][h][d] from 32 fp32 accumulator columns
// times mul (nullptr: zeros). A warp's lanes write 64 contiguous bytes per query.
__device__ __forceinline__ void store_chunk_cols(__nv_bfloat16* out, int64_t q_first, int nq, int H, int h, int d,
                                                 int c0, const uint32_t* v, float mul) {
  for (int e = 0; e < 32; ++e) {
    const int q = c0 + e;
    if (q >= nq) break;
    const float x = v ? __uint_as_float(v[e]) * mul : 0.0f;
    out[((q_first + q) * H + h) * kD + d] = __float2bfloat16_rn(x);
  }
}

// P^T / dS^T as bf16 A operands: activation warpgroup g packs its 32 query
// columns over the first 16 of its own 32 fp32 columns (hi parts) and the
// next 16 (lo parts), so neither warpgroup writes where the other still
// reads; the kk-th 16-query slice of the hi parts sits at a_col(kk).
__device__ __forceinline__ uint32_t a_col(int kk) { return static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8); }

// ---------------------------------------------------------------------------- short-key forward
// Cross-attention over short key sequences (every sequence at most 128 keys):
// one item = (sequence, head) with all of its 128-row query tiles, in the
// usual orientation (S = Q K^T, M = queries). The item's one K / V tile is
// loaded once; its query tiles stream through a 4-stage ring, and the two
// activation warpgroups take alternate tiles: S and O are double-buffered in
// TMEM ([S0 | S1 | O0 | O1]), so one warpgroup's activation and epilogue
// overlap the other's products. With a single key tile O = P V needs no
// online accumulation: the product overwrites O.
constexpr int kSkvQStages = 4;
constexpr int kSkvCtlRegs = 104;  // 384 x 168 at launch = 128 x 104 + 256 x 200
constexpr int kSkvActRegs = 200;
static_assert(128 * kSkvCtlRegs + 256 * kSkvActRegs <= kThreads * 168, "register split");

template <bool HILO>
struct SfCfg {
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;  // stage s at kQOff + s * kTileBytes
  static constexpr int kBarOff = kQOff + kSkvQStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256;
  static constexpr uint32_t kOCol = 2 * kTile;  // S_g at g * 128, O_g at kOCol + g * 128
};
static_assert(SfCfg<false>::kSmemBytes <= 227 * 1024, "shared memory");

struct SfBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[kSkvQStages], q_empty[kSkvQStages];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(SfBars) <= 256, "barrier block overflows its slot");

template <int ACT, bool HILO>
__global__ void __launch_bounds__(kThreads, 1)
    skv_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnArgs a, const int* gate) {
  using C = SfCfg<HILO>;
  if (*gate == 0) return;  // some sequence holds more than 128 keys: the general forward runs
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(a.status, JATTN_ERR_UNSUPPORTED, 110, blockIdx.x);
    return;
  }
  uint8_t* sm = smem_raw;
  SfBars* bars = reinterpret_cast<SfBars*>(sm + C::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int s = 0; s < kSkvQStages; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&bars->s_full[g], 1);
      mbar_init(&bars->p_full[g], kTile);
      mbar_init(&bars->o_full[g], 1);
      mbar_init(&bars->o_empty[g], kTile);
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
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSkvCtlRegs));
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t kv_it = 0, q_it = 0;
      bool ok = true, kv_armed = false;
      // the item's K / V copy is skipped under debug flag bit 1, so that the
      // waits for it time out
      const bool skip = (a.debug_flags & 1) != 0;
      PItem it;
      for (long long r = 0; ok && load_bitem<true>(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->kv_empty, (kv_it & 1) ^ 1, abort_flag, a, 111))) break;
        if (!skip) {
          mbar_arrive_expect_tx(&bars->kv_full, 2 * kTileBytes);
          for (int c = 0; c < 2; ++c) {
            tma_load_2d(sm + C::kKOff + c * kBoxK, &tmK, &bars->kv_full, it.h * kD + c * 64, static_cast<int>(it.k0));
            tma_load_2d(sm + C::kVOff + c * kBoxK, &tmV, &bars->kv_full, it.h * kD + c * 64, static_cast<int>(it.k0));
          }
          kv_armed = true;
        }
        ++kv_it;
        for (int t = it.lo; t < it.hi && ok; ++t, ++q_it) {
          const int s = q_it % kSkvQStages;
          if (!(ok = wait_bar(&bars->q_empty[s], ((q_it / kSkvQStages) & 1) ^ 1, abort_flag, a, 112))) break;
          mbar_arrive_expect_tx(&bars->q_full[s], kTileBytes);
          for (int c = 0; c < 2; ++c)
            tma_load_2d(sm + C::kQOff + s * kTileBytes + c * kBoxK, &tmQ, &bars->q_full[s], it.h * kD + c * 64,
                        static_cast<int>(it.q0) + t * kTile);
        }
      }
      if (kv_armed) drain_wait(&bars->kv_full, (kv_it - 1) & 1, a.timeout_ns);
      for (uint32_t i = (q_it > (uint32_t)kSkvQStages ? q_it - kSkvQStages : 0); i < q_it; ++i)
        drain_wait(&bars->q_full[i % kSkvQStages], (i / kSkvQStages) & 1, a.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kTile, kTile, false, false);  // S = Q K^T
      constexpr uint32_t idO = idesc_bf16_f32(kTile, kD, false, true);      // O = P V
      const uint64_t dK = sdesc_sw128(smem_u32(sm + C::kKOff), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(sm + C::kVOff), kBoxK, 1024);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(sm + C::kQOff), 16, 1024);
      uint32_t kv_it = 0, q_used = 0, n = 0;
      bool ok = true;
      PItem it;
      // O_g = P_g V for the item's t-th query tile (global tile nt)
      auto issue_pv = [&](uint32_t nt) -> bool {
        const uint32_t g = nt & 1, u = nt >> 1;
        if (!wait_bar(&bars->p_full[g], u & 1, abort_flag, a, 113)) return false;
        if (!wait_bar(&bars->o_empty[g], (u & 1) ^ 1, abort_flag, a, 114)) return false;
        tc_fence_after();
        constexpr int kNP = HILO ? 2 : 1;
#pragma unroll
        for (int hl = 0; hl < kNP; ++hl)
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ts(tmem + C::kOCol + g * kD, tmem + g * kTile + 64 * hl + kk * 8, dV + mnslice(kk), idO,
                   (hl > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->o_full[g]);
        return true;
      };
      for (long long r = 0; ok && load_bitem<true>(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->kv_full, kv_it & 1, abort_flag, a, 115))) break;
        ++kv_it;
        const int nq = it.hi - it.lo;
        for (int t = 0; t < nq && ok; ++t) {
          const uint32_t nt = n + t, g = nt & 1, qi = q_used + t;
          const int qs = qi % kSkvQStages;
          if (!(ok = wait_bar(&bars->q_full[qs], (qi / kSkvQStages) & 1, abort_flag, a, 116))) break;
          tc_fence_after();
          // S_g overwrites P_g of tile nt - 2, which its PV product (issued
          // before) has read
          const uint64_t qd = dQ0 + qs * (kTileBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            mma_ss(tmem + g * kTile, qd + kslice(kk, kBoxK), dK + kslice(kk, kBoxK), idS, kk > 0 ? 1u : 0u);
          mma_commit(&bars->s_full[g]);
          mma_commit(&bars->q_empty[qs]);
          if (t > 0) ok = issue_pv(nt - 1);
        }
        if (ok) ok = issue_pv(n + nq - 1);
        if (!ok) break;
        mma_commit(&bars->kv_empty);  // K read by the S products, V by the PV products
        n += nq;
        q_used += nq;
      }
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, a.timeout_ns);
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSkvActRegs));
    // ------------------------------------------------------------ activation warpgroups
    // Warpgroup g takes the query tiles of global index g mod 2: its S_g
    // becomes P_g (bf16 hi parts over S_g's first 64 columns, lo parts over
    // the next 64), then it stores O_g's rows.
    const int g = (warp - 4) >> 2;
    const int row = 32 * (warp & 3) + lane;  // query row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + g * kTile, tO = tmem + lane_base + C::kOCol + g * kD;
    uint32_t n = 0;
    bool ok = true;
    PItem it;
    for (long long r = 0; ok && load_bitem<true>(a, r, it); ++r) {
      const int nq = it.hi - it.lo;
      if (nq <= 0) continue;  // no queries: nothing to write (the gate admits no queries without keys)
      const float cn = (a.norm_by_lkv && it.lkv > 0) ? 1.0f / it.lkv : 1.0f;
      const int nkc = (it.lkv + 31) / 32;  // 32-key chunks that hold keys
      for (int t = 0; t < nq; ++t) {
        const uint32_t nt = n + t;
        if ((nt & 1) != static_cast<uint32_t>(g)) continue;
        const uint32_t u = nt >> 1;
        ok = __all_sync(0xffffffffu, wait_bar(&bars->s_full[g], u & 1, abort_flag, a, 117));
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[kTile];
#pragma unroll
        for (int c = 0; c < kTile / 32; ++c)
          if (c < nkc) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c));
        tmem_ld_wait();
        // P over the keys of the sequence; zero past its end (V rows there
        // belong to other sequences)
#pragma unroll
        for (int c = 0; c < kTile / 32; ++c) {
          uint32_t hi[16], lo[16];
          if (c < nkc) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int kc = 32 * c + 2 * e;
              const float f0 = kc < it.lkv ? act_f<ACT>(__uint_as_float(sv[kc]) * a.scale) : 0.0f;
              const float f1 = kc + 1 < it.lkv ? act_f<ACT>(__uint_as_float(sv[kc + 1]) * a.scale) : 0.0f;
              hi[e] = pack_bf16x2(f0, f1);
              if constexpr (HILO) lo[e] = bf16x2_lo(f0, f1, hi[e]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) hi[e] = lo[e] = 0u;
          }
          tmem_st16(tS + 16 * c, hi);
          if constexpr (HILO) tmem_st16(tS + 64 + 16 * c, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_full[g]);
        // O_g = P_g V, times 1/Lkv when asked, to the tile's rows of the sequence
        ok = __all_sync(0xffffffffu, wait_bar(&bars->o_full[g], u & 1, abort_flag, a, 118));
        if (!ok) break;
        tc_fence_after();
        const int ql = (it.lo + t) * kTile + row;
        const bool valid = ql < it.lq;
        __nv_bfloat16* orow = a.out0 + ((it.q0 + ql) * a.H + it.h) * kD;
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tO + 32 * c, v);
          tmem_ld_wait();
          if (c == kD / 32 - 1) {
            tc_fence_before();
            mbar_arrive(&bars->o_empty[g]);
          }
          if (valid) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * cn, __uint_as_float(v[2 * e + 1]) * cn);
            store_words16(orow + 32 * c, w, a.out_v8);
          }
        }
      }
      if (!ok) break;
      n += nq;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------- short-key backward
// Cross-attention over short key sequences, backward, with 128 queries per
// step so that every product runs at N = 128. One item = (sequence, head):
// its K / V tile stays in shared memory, its 128-row Q / dO tiles stream
// through a 2-stage ring. Per step (query tile t):
//   S^T = K Q^T, dP^T = V dO^T            (TMEM lanes = keys)
//   P^T, dS^T = act'(scale S^T) * dP^T     (bf16, back into TMEM as A operands)
//   dV += P^T dO, dK += dS^T Q             (accumulated over the item)
//   dQ = dS K                              (A = dS^T from shared memory, MN-major;
//                                           into the dP^T columns once dK has
//                                           read dS^T: lanes = queries)
// and the epilogue warpgroup writes dQ's rows each step and dK / dV's rows at
// the item's end. TMEM [S^T | dP^T, then dQ | dV | dK] = 512 columns; the next
// step's S^T is issued right after this step's dQ, its dP^T once the
// epilogue has read dQ. dS^T reaches TMEM first (dK may start) and the shared
// tile second (dQ waits for it); the epilogue stages dQ's rows as bf16 in that
// tile's room once dQ has read it, stores them row-coalesced, and only then
// lets the activation write the next step's dS^T there. Warps whose 32 key
// rows all lie past the item's keys skip the activation and write zeros.
constexpr int kSbCtlRegs = 128;  // 512 x 128 at launch = 128 x (128 + 2 x 160 + 64)
constexpr int kSbActRegs = 160;
constexpr int kSbEpiRegs = 64;
static_assert(128 * (kSbCtlRegs + 2 * kSbActRegs + kSbEpiRegs) <= kBwdThreads * 128, "register split");
constexpr int kSbMaxStages = 2;

// setmaxnreg toward R registers from the 128 at launch: .inc above, .dec below.
template <int R>
__device__ __forceinline__ void sb_set_regs() {
  if constexpr (R > 128) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
  if constexpr (R < 128) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

template <bool HILO>
struct SbCfg {
  static constexpr int kStages = HILO ? 1 : 2;  // Q / dO ring (the hi + lo dS^T tiles take the second stage's room)
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQDOff = 2 * kTileBytes;  // stage s: Q tile, then dO tile
  static constexpr int kNP = HILO ? 2 : 1;
  static constexpr int kDSOff = kQDOff + kStages * 2 * kTileBytes;  // dS^T [keys][queries] (hi, lo)
  static constexpr int kBarOff = kDSOff + kNP * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256;
  static constexpr uint32_t kSCol = 0, kDPCol = 128, kDVCol = 256, kDKCol = 384;  // dQ over kDPCol
};
static_assert(SbCfg<false>::kSmemBytes <= 227 * 1024 && SbCfg<true>::kSmemBytes <= 227 * 1024, "shared memory");

struct SbBars {
  uint64_t kv_full, kv_empty;
  uint64_t qd_full[kSbMaxStages], qd_empty[kSbMaxStages];
  uint64_t s_full, dp_full, p_ready, ds_ready, dsm_free;
  uint64_t acc_full, acc_empty, dq_full, dq_empty, drain, epi_sync, dsm_ready;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(SbBars) <= 256, "barrier block overflows its slot");

// A operand column of the kk-th 16-query slice (hi parts hl = 0, lo parts
// hl = 1) of P^T / dS^T: activation warpgroup g owns fp32 columns
// [64 g, 64 g + 64) and packs each 32-query half in place of its own 32
// columns, hi parts over the first 16 and lo parts over the next 16.
__device__ __forceinline__ uint32_t sb_acol(int kk, int hl) {
  return static_cast<uint32_t>((kk >> 2) * 64 + ((kk >> 1) & 1) * 32 + hl * 16 + (kk & 1) * 8);
}

// 16 packed bf16 pairs (queries c0 .. c0 + 31 of key row `row`) into a
// [128 keys][128 queries] tile made of two [128][64] 128-byte-swizzled boxes.
__device__ __forceinline__ void st_dst_row(uint32_t tile, int row, int c0, const uint32_t (&w)[16]) {
  st_pt_row(tile + (c0 >> 6) * kBoxK, row, c0 & 63, w);
}

template <int ACT, bool HILO>
__global__ void __launch_bounds__(kBwdThreads, 1)
    skv_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                   const AttnArgs a, const int* gate) {
  using C = SbCfg<HILO>;
  if (*gate == 0) return;  // some sequence holds more than 128 keys: the general passes run
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(a.status, JATTN_ERR_UNSUPPORTED, 120, blockIdx.x);
    return;
  }
  uint8_t* sm = smem_raw;
  SbBars* bars = reinterpret_cast<SbBars*>(sm + C::kBarOff);
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
    mbar_init(&bars->p_ready, 2 * kTile);
    mbar_init(&bars->ds_ready, 2 * kTile);
    mbar_init(&bars->dsm_ready, 2 * kTile);
    mbar_init(&bars->dsm_free, kTile);  // the epilogue has stored the dQ rows staged there
    mbar_init(&bars->epi_sync, kTile);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, kTile);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, kTile);
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
  sb_set_regs<kSbCtlRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      uint32_t kv_it = 0, qd_it = 0;
      bool ok = true, kv_armed = false;
      const bool skip = (a.debug_flags & 1) != 0;  // the item's K / V copy, so that its waits time out
      PItem it;
      for (long long r = 0; ok && load_bitem<true>(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        // the item's first Q / dO copies go out before its K / V copy, which
        // waits for the item before to finish
        auto load_kv = [&]() -> bool {
          if (!wait_bar(&bars->kv_empty, (kv_it & 1) ^ 1, abort_flag, a, 121)) return false;
          if (!skip) {
            mbar_arrive_expect_tx(&bars->kv_full, 2 * kTileBytes);
            for (int c = 0; c < 2; ++c) {
              tma_load_2d(sm + C::kKOff + c * kBoxK, &tmK, &bars->kv_full, it.h * kD + c * 64,
                          static_cast<int>(it.k0));
              tma_load_2d(sm + C::kVOff + c * kBoxK, &tmV, &bars->kv_full, it.h * kD + c * 64,
                          static_cast<int>(it.k0));
            }
            kv_armed = true;
          }
          ++kv_it;
          return true;
        };
        const int pre = min(it.hi - it.lo, C::kStages);
        for (int t = it.lo; t < it.hi && ok; ++t, ++qd_it) {
          if (t == it.lo + pre && !(ok = load_kv())) break;
          const int s = qd_it % C::kStages;
          if (!(ok = wait_bar(&bars->qd_empty[s], ((qd_it / C::kStages) & 1) ^ 1, abort_flag, a, 122))) break;
          mbar_arrive_expect_tx(&bars->qd_full[s], 2 * kTileBytes);
          uint8_t* dst = sm + C::kQDOff + s * 2 * kTileBytes;
          const int y = static_cast<int>(it.q0) + t * kTile;
          for (int c = 0; c < 2; ++c) {
            tma_load_2d(dst + c * kBoxK, &tmQ, &bars->qd_full[s], it.h * kD + c * 64, y);
            tma_load_2d(dst + kTileBytes + c * kBoxK, &tmDO, &bars->qd_full[s], it.h * kD + c * 64, y);
          }
        }
        if (ok && pre == it.hi - it.lo) ok = load_kv();
      }
      if (kv_armed) drain_wait(&bars->kv_full, (kv_it - 1) & 1, a.timeout_ns);
      for (uint32_t i = (qd_it > (uint32_t)C::kStages ? qd_it - C::kStages : 0); i < qd_it; ++i)
        drain_wait(&bars->qd_full[i % C::kStages], (i / C::kStages) & 1, a.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kTile, kTile, false, false);  // S^T = K Q^T, dP^T = V dO^T
      constexpr uint32_t idG = idesc_bf16_f32(kTile, kD, false, true);      // dV = P^T dO, dK = dS^T Q
      constexpr uint32_t idQ = idesc_bf16_f32(kTile, kD, true, true);       // dQ = dS K
      const uint32_t sK = smem_u32(sm + C::kKOff), sV = smem_u32(sm + C::kVOff), sQD = smem_u32(sm + C::kQDOff);
      const uint64_t dKk = sdesc_sw128(sK, 16, 1024), dVk = sdesc_sw128(sV, 16, 1024);
      const uint64_t dKm = sdesc_sw128(sK, kBoxK, 1024);
      const uint64_t dDS = sdesc_sw128(smem_u32(sm + C::kDSOff), kBoxK, 1024);
      uint32_t kv_it = 0, qd_used = 0, acc_n = 0, n = 0;
      bool ok = true;
      PItem it;
      auto qbase = [&](uint32_t qi) { return sQD + (qi % C::kStages) * 2 * kTileBytes; };
      // S^T of step t (query tile qi)
      auto issue_s = [&](uint32_t qi) -> bool {
        const int qs = qi % C::kStages;
        if (!wait_bar(&bars->qd_full[qs], (qi / C::kStages) & 1, abort_flag, a, 123)) return false;
        tc_fence_after();
        const uint64_t dQk = sdesc_sw128(qbase(qi), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem + C::kSCol, dKk + kslice(kk, kBoxK), dQk + kslice(kk, kBoxK), idS, kk > 0 ? 1u : 0u);
        mma_commit(&bars->s_full);
        return true;
      };
      // dP^T of step t (overwrites the dQ of the step before, once read)
      auto issue_dp = [&](uint32_t qi, uint32_t nt) -> bool {
        if (!wait_bar(&bars->dq_empty, (nt & 1) ^ 1, abort_flag, a, 124)) return false;
        tc_fence_after();
        const uint64_t dDOk = sdesc_sw128(qbase(qi) + kTileBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem + C::kDPCol, dVk + kslice(kk, kBoxK), dDOk + kslice(kk, kBoxK), idS, kk > 0 ? 1u : 0u);
        mma_commit(&bars->dp_full);
        return true;
      };
      for (long long r = 0; ok && load_bitem<true>(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        if (!(ok = wait_bar(&bars->kv_full, kv_it & 1, abort_flag, a, 125))) break;
        ++kv_it;
        tc_fence_after();
        const int ns = it.hi - it.lo;
        if (!(ok = issue_s(qd_used) && issue_dp(qd_used, n))) break;
        for (int t = 0; t < ns; ++t) {
          const uint32_t nt = n + t, qi = qd_used + t;
          const uint32_t qb = qbase(qi);
          const uint64_t dQm = sdesc_sw128(qb, kBoxK, 1024), dDOm = sdesc_sw128(qb + kTileBytes, kBoxK, 1024);
          // dV += P^T dO, once P^T is in TMEM (and, on the item's first step,
          // the epilogue has drained the item before's dV / dK)
          if (!(ok = wait_bar(&bars->p_ready, nt & 1, abort_flag, a, 126))) break;
          if (t == 0 && !(ok = wait_bar(&bars->acc_empty, (acc_n & 1) ^ 1, abort_flag, a, 127))) break;
          tc_fence_after();
#pragma unroll
          for (int hl = 0; hl < C::kNP; ++hl)
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ts(tmem + C::kDVCol, tmem + C::kSCol + sb_acol(kk, hl), dDOm + mnslice(kk), idG,
                     (t > 0 || hl > 0 || kk > 0) ? 1u : 0u);
          if (!(ok = wait_bar(&bars->ds_ready, nt & 1, abort_flag, a, 128))) break;
          tc_fence_after();
#pragma unroll
          for (int hl = 0; hl < C::kNP; ++hl)
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ts(tmem + C::kDKCol, tmem + C::kDPCol + sb_acol(kk, hl), dQm + mnslice(kk), idG,
                     (t > 0 || hl > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars->qd_empty[qi % C::kStages]);  // dK was the last product to read Q / dO
          if (!(ok = wait_bar(&bars->dsm_ready, nt & 1, abort_flag, a, 135))) break;
          // dQ = dS K into the dP^T columns (dK has been issued: in order, it
          // reads dS^T first); then the shared dS^T tile is free
#pragma unroll
          for (int hl = 0; hl < C::kNP; ++hl)
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ss(tmem + C::kDPCol, dDS + hl * (kTileBytes >> 4) + mnslice(kk), dKm + mnslice(kk), idQ,
                     (hl > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars->dq_full);
          if (t + 1 < ns) {
            if (!(ok = issue_s(qi + 1))) break;
            if (!(ok = issue_dp(qi + 1, nt + 1))) break;
          }
        }
        if (!ok) break;
        mma_commit(&bars->acc_full);
        ++acc_n;
        mma_commit(&bars->kv_empty);
        n += ns;
        qd_used += ns;
      }
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, a.timeout_ns);
    }
    __syncwarp();
  }
  } else if (warp < 12) {
    sb_set_regs<kSbActRegs>();
    // ------------------------------------------------------------ activation warpgroups
    // warpgroup g takes queries [64 g, 64 g + 64) of every step
    const int g = (warp - 4) >> 2;
    const int row = 32 * (warp & 3) + lane;  // key row
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + C::kSCol + 64 * g, tDP = tmem + lane_base + C::kDPCol + 64 * g;
    const uint32_t sDS = smem_u32(sm + C::kDSOff);
    uint32_t n = 0;
    bool ok = true;
    PItem it;
    for (long long r = 0; ok && load_bitem<true>(a, r, it); ++r) {
      if (it.hi <= it.lo) continue;
      const int ns = it.hi - it.lo;
      const bool valid = row < it.lkv;
      const bool live = 32 * (warp & 3) < it.lkv;  // the warp holds one of the item's key rows
      for (int t = 0; t < ns; ++t) {
        const uint32_t nt = n + t;
        const int nq = min(kTile, it.lq - (it.lo + t) * kTile) - 64 * g;  // this group's query columns
        ok = __all_sync(0xffffffffu, wait_bar(&bars->s_full, nt & 1, abort_flag, a, 129));
        if (!ok) break;
        tc_fence_after();
        // One 32-column half at a time, so that only the derivatives stay live
        // across the dP^T wait; each half's hi and lo parts go in place of
        // its own 32 columns. A warp whose 32 key rows all lie past the
        // item's keys computes nothing and writes zeros. P^T rows of keys
        // past the end are left unmasked (they reach only dV rows that are
        // never stored); dS^T rows are masked, since dQ sums over keys.
        float gr[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t hi[16], lo[16];
          if (live && 32 * c < nq) {
            uint32_t sv[32];
            tmem_ld32(tS + 32 * c, sv);
            tmem_ld_wait();
            if (32 * c + 32 <= nq) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float f0, f1;
                act_and_grad<ACT>(__uint_as_float(sv[2 * e]) * a.scale, f0, gr[32 * c + 2 * e]);
                act_and_grad<ACT>(__uint_as_float(sv[2 * e + 1]) * a.scale, f1, gr[32 * c + 2 * e + 1]);
                hi[e] = pack_bf16x2(f0, f1);
                if constexpr (HILO) lo[e] = bf16x2_lo(f0, f1, hi[e]);
              }
            } else {  // the item's last query tile: columns past its queries are zero
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int q = 32 * c + 2 * e;
                float f0, f1, g0, g1;
                act_and_grad<ACT>(__uint_as_float(sv[2 * e]) * a.scale, f0, g0);
                act_and_grad<ACT>(__uint_as_float(sv[2 * e + 1]) * a.scale, f1, g1);
                const bool a0 = q < nq, a1 = q + 1 < nq;
                f0 = a0 ? f0 : 0.0f;
                f1 = a1 ? f1 : 0.0f;
                gr[q] = a0 ? g0 : 0.0f;
                gr[q + 1] = a1 ? g1 : 0.0f;
                hi[e] = pack_bf16x2(f0, f1);
                if constexpr (HILO) lo[e] = bf16x2_lo(f0, f1, hi[e]);
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) hi[e] = lo[e] = 0u;
          }
          tmem_st16(tS + 32 * c, hi);
          if constexpr (HILO) tmem_st16(tS + 32 * c + 16, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_ready);

        ok = __all_sync(0xffffffffu, wait_bar(&bars->dp_full, nt & 1, abort_flag, a, 130));
        if (!ok) break;
        tc_fence_after();
        // dS^T into TMEM first (dK may start), then, once the epilogue has
        // stored the step before's dQ rows from the shared tile's room, into
        // the shared tile (dQ may start)
        uint32_t hh[2][16], ll[2][16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (live && 32 * c < nq) {
            uint32_t dv[32];
            tmem_ld32(tDP + 32 * c, dv);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int q = 32 * c + 2 * e;
              const float d0 = gr[q] * __uint_as_float(dv[2 * e]), d1 = gr[q + 1] * __uint_as_float(dv[2 * e + 1]);
              hh[c][e] = valid ? pack_bf16x2(d0, d1) : 0u;
              if constexpr (HILO) ll[c][e] = valid ? bf16x2_lo(d0, d1, hh[c][e]) : 0u;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) hh[c][e] = ll[c][e] = 0u;
          }
          tmem_st16(tDP + 32 * c, hh[c]);
          if constexpr (HILO) tmem_st16(tDP + 32 * c + 16, ll[c]);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->ds_ready);
        ok = __all_sync(0xffffffffu, wait_bar(&bars->dsm_free, (nt & 1) ^ 1, abort_flag, a, 131));
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          st_dst_row(sDS, row, 64 * g + 32 * c, hh[c]);
          if constexpr (HILO) st_dst_row(sDS + kTileBytes, row, 64 * g + 32 * c, ll[c]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->dsm_ready);
      }
      if (!ok) break;
      n += ns;
    }
  } else {
    sb_set_regs<kSbEpiRegs>();
    // ------------------------------------------------------------ epilogue warpgroup
    // dQ rows (thread = query row) every step, dV / dK rows (thread = key row)
    // at the item's end; items without queries get zero dK / dV rows.
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t sDQ = smem_u32(sm + C::kDSOff);
    uint32_t acc_n = 0, n = 0;
    bool ok = true;
    PItem it;
    for (long long r = 0; ok && load_bitem<true>(a, r, it); ++r) {
      const bool kvalid = row < it.lkv;
      const int64_t gk = it.k0 + row;
      __nv_bfloat16* dv_row = a.out1 + (gk * a.H + it.h) * kD;
      __nv_bfloat16* dk_row = a.out2 + (gk * a.H + it.h) * kD;
      if (it.hi <= it.lo) {
        if (kvalid) {
          uint4* dv = reinterpret_cast<uint4*>(dv_row);
          uint4* dk = reinterpret_cast<uint4*>(dk_row);
          for (int e = 0; e < kD / 8; ++e) dv[e] = dk[e] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int ns = it.hi - it.lo;
      const float cn = (a.norm_by_lkv && it.lkv > 0) ? 1.0f / it.lkv : 1.0f;
      for (int t = 0; t < ns && ok; ++t) {
        const uint32_t nt = n + t;
        ok = __all_sync(0xffffffffu, wait_bar(&bars->dq_full, nt & 1, abort_flag, a, 132));
        if (!ok) break;
        tc_fence_after();
        // dQ's rows (thread = query row) as bf16 into the dS^T tile's room,
        // which the dQ product has finished reading: row r at r * 256 bytes,
        // its 16-byte piece p at p ^ (r & 7). The TMEM columns are released
        // after the last load, before any global store.
        const float mul = cn * a.scale;
#pragma unroll 1
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + C::kDPCol + 32 * c, v);
          tmem_ld_wait();
          if (c == kD / 32 - 1) {
            tc_fence_before();
            mbar_arrive(&bars->dq_empty);
          }
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
          const uint32_t rb = sDQ + static_cast<uint32_t>(row) * 256;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_shared_v4(rb + (((4 * c + i) ^ (row & 7)) << 4), w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
        // all 128 rows staged; then warp w stores rows 32 w .. 32 w + 31, two
        // 256-byte rows per instruction, and the tile's room goes back to the
        // activation
        mbar_arrive(&bars->epi_sync);
        ok = __all_sync(0xffffffffu, wait_bar(&bars->epi_sync, nt & 1, abort_flag, a, 134));
        if (!ok) break;
        const int q_tile0 = (it.lo + t) * kTile;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          const int r = 32 * (warp & 3) + 2 * i + (lane >> 4), pc = lane & 15;
          const uint4 val = ld_shared_v4(sDQ + static_cast<uint32_t>(r) * 256 + ((pc ^ (r & 7)) << 4));
          const int ql = q_tile0 + r;
          if (ql < it.lq) *reinterpret_cast<uint4*>(a.out0 + ((it.q0 + ql) * a.H + it.h) * kD + 8 * pc) = val;
        }
        mbar_arrive(&bars->dsm_free);
      }
      if (!ok) break;
      n += ns;
      ok = __all_sync(0xffffffffu, wait_bar(&bars->acc_full, acc_n & 1, abort_flag, a, 133));
      if (!ok) break;
      ++acc_n;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 2 * kD / 32; ++c) {
        const bool is_dk = c >= kD / 32;
        const int cc = is_dk ? c - kD / 32 : c;
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + (is_dk ? C::kDKCol : C::kDVCol) + 32 * cc, v);
        tmem_ld_wait();
        if (c == 2 * kD / 32 - 1) {
          tc_fence_before();
          mbar_arrive(&bars->acc_empty);
        }
        if (kvalid) {
          uint32_t w[16];
          const float mul = is_dk ? cn * a.scale : cn;
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
          store_words16((is_dk ? dk_row : dv_row) + 32 * cc, w, a.out_v8);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------- backward
// Two modes share the kernel. Pooling (CROSS = false): an item is (sequence,
// head) with at most 64 queries, loaded once, and its key tiles are the steps;
// dV and dK are complete per step, dQ^T accumulates over the item. Cross
// attention over short key sequences (CROSS = true): an item is (sequence,
// head) with at most 128 keys, loaded once, and its 64-query chunks are the
// steps; dQ^T is complete per step, dV and dK accumulate over the item.
template <bool HILO, bool CROSS>
struct PbCfg {
  static constexpr int kQDStages = CROSS ? 4 : 1;  // Q + dO chunk pairs
  static constexpr int kKStages = CROSS ? 1 : 3;
  static constexpr int kVStages = CROSS ? 1 : 2;
  static constexpr int kNP = HILO ? 2 : 1;  // dS^T tiles in shared memory (hi, lo)
  static constexpr int kQDOff = 0;          // stage s: Q chunk, then dO chunk
  static constexpr int kKOff = kQDStages * 2 * kChunkBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kDSOff = kVOff + kVStages * kTileBytes;
  static constexpr int kBarOff = kDSOff + kNP * kPBytes;
  static constexpr int kSmemBytes = kBarOff + 256;
  // TMEM: S^T (P^T as bf16 over its first columns), dP^T (dS^T likewise), dV, dK, dQ^T
  static constexpr uint32_t kSCol = 0, kDPCol = 64, kDVCol = 128, kDKCol = 256, kDQCol = 384;
};
static_assert(PbCfg<false, false>::kSmemBytes <= 227 * 1024 && PbCfg<true, false>::kSmemBytes <= 227 * 1024 &&
                  PbCfg<false, true>::kSmemBytes <= 227 * 1024 && PbCfg<true, true>::kSmemBytes <= 227 * 1024,
              "shared memory");

struct PbBars {
  uint64_t qd_full[4], qd_empty[4];  // Q and dO chunks
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full, dp_full, p_ready, ds_ready, dsm_free;
  uint64_t acc_full, acc_empty, dq_full, dq_empty, drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(PbBars) <= 256, "barrier block overflows its slot");

template <int ACT, bool HILO, bool CROSS>
__global__ void __launch_bounds__(kBwdThreads, 1)
    pma_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                   const AttnArgs a, const int* gate) {
  using C = PbCfg<HILO, CROSS>;
  if (*gate == 0) return;  // some sequence is outside this mode's limits: the general passes run
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(a.status, JATTN_ERR_UNSUPPORTED, 93, blockIdx.x);
    return;
  }
  uint8_t* sm = smem_raw;
  PbBars* bars = reinterpret_cast<PbBars*>(sm + C::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &bars->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kQDStages; ++s) {
      mbar_init(&bars->qd_full[s], 1);
      mbar_init(&bars->qd_empty[s], 1);
    }
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, 2 * kTile);
    mbar_init(&bars->ds_ready, 2 * kTile);
    mbar_init(&bars->dsm_free, 1);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, kTile);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, kTile);
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
  // each warpgroup sets its register share in the branch that holds its code
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kCtlRegs));
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      uint32_t k_it = 0, v_it = 0, qd_it = 0;
      bool ok = true;
      PItem it;
      // the copy an item loads once (pooling: Q and dO; cross: K and V) is
      // skipped under debug flag bit 1, so that the waits for it time out
      const bool skip_once = (a.debug_flags & 1) != 0;
      auto load_kv = [&](const CUtensorMap* map, uint64_t* full, uint64_t* empty, int stages, int off, uint32_t& cnt,
                         int j, int where, bool skip) -> bool {
        const int s = cnt % stages;
        if (!wait_bar(&empty[s], ((cnt / stages) & 1) ^ 1, abort_flag, a, where)) return false;
        if (!skip) {
          mbar_arrive_expect_tx(&full[s], kTileBytes);
          for (int c = 0; c < 2; ++c)
            tma_load_2d(sm + off + s * kTileBytes + c * kBoxK, map, &full[s], it.h * kD + c * 64,
                        static_cast<int>(it.k0) + j * kTile);
        }
        ++cnt;
        return true;
      };
      auto load_qd = [&](int64_t row, bool skip) -> bool {
        const int s = qd_it % C::kQDStages;
        if (!wait_bar(&bars->qd_empty[s], ((qd_it / C::kQDStages) & 1) ^ 1, abort_flag, a, 94)) return false;
        if (!skip) {
          mbar_arrive_expect_tx(&bars->qd_full[s], 2 * kChunkBytes);
          uint8_t* dst = sm + C::kQDOff + s * 2 * kChunkBytes;
          for (int c = 0; c < 2; ++c) {
            tma_load_2d(dst + c * kBoxQ, &tmQ, &bars->qd_full[s], it.h * kD + c * 64, static_cast<int>(row));
            tma_load_2d(dst + kChunkBytes + c * kBoxQ, &tmDO, &bars->qd_full[s], it.h * kD + c * 64,
                        static_cast<int>(row));
          }
        }
        ++qd_it;
        return true;
      };
      for (long long r = 0; ok && load_bitem<CROSS>(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        if constexpr (CROSS) {
          if (!(ok = load_kv(&tmK, bars->k_full, bars->k_empty, 1, C::kKOff, k_it, it.rt, 95, skip_once))) break;
          if (!(ok = load_kv(&tmV, bars->v_full, bars->v_empty, 1, C::kVOff, v_it, it.rt, 96, skip_once))) break;
          for (int c = it.lo; c < it.hi && ok; ++c) ok = load_qd(it.q0 + static_cast<int64_t>(c) * kQC, false);
        } else {
          if (!(ok = load_qd(it.q0, skip_once))) break;
          for (int j = it.lo; j < it.hi && ok; ++j) {
            if (!(ok = load_kv(&tmK, bars->k_full, bars->k_empty, C::kKStages, C::kKOff, k_it, j, 95, false))) break;
            ok = load_kv(&tmV, bars->v_full, bars->v_empty, C::kVStages, C::kVOff, v_it, j, 96, false);
          }
        }
      }
      // every copy this thread started lands before the CTA can exit (skipped
      // copies started nothing)
      if (!(skip_once && !CROSS))
        for (uint32_t i = (qd_it > (uint32_t)C::kQDStages ? qd_it - C::kQDStages : 0); i < qd_it; ++i)
          drain_wait(&bars->qd_full[i % C::kQDStages], (i / C::kQDStages) & 1, a.timeout_ns);
      if (!(skip_once && CROSS)) {
        for (uint32_t i = (k_it > (uint32_t)C::kKStages ? k_it - C::kKStages : 0); i < k_it; ++i)
          drain_wait(&bars->k_full[i % C::kKStages], (i / C::kKStages) & 1, a.timeout_ns);
        for (uint32_t i = (v_it > (uint32_t)C::kVStages ? v_it - C::kVStages : 0); i < v_it; ++i)
          drain_wait(&bars->v_full[i % C::kVStages], (i / C::kVStages) & 1, a.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kTile, kQC, false, false);  // S^T = K Q^T, dP^T = V dO^T
      constexpr uint32_t idG = idesc_bf16_f32(kTile, kD, false, true);    // dV = P^T dO, dK = dS^T Q
      constexpr uint32_t idQ = idesc_bf16_f32(kD, kQC, true, true);       // dQ^T += K^T dS^T
      const uint32_t sQD = smem_u32(sm + C::kQDOff);
      const uint32_t sK = smem_u32(sm + C::kKOff), sV = smem_u32(sm + C::kVOff), sDS = smem_u32(sm + C::kDSOff);
      const uint64_t dK0 = sdesc_sw128(sK, 16, 1024), dKt0 = sdesc_sw128(sK, kBoxK, 1024);
      const uint64_t dV0 = sdesc_sw128(sV, 16, 1024), dDS0 = sdesc_sw128(sDS, kPBytes, 1024);
      uint32_t k_used = 0, v_used = 0, qd_used = 0, acc_n = 0, dq_n = 0, n = 0;
      bool ok = true;
      PItem it;
      // stages of step t's tiles: key tile (ks, vs) and query chunk (qs)
      auto k_idx = [&](int t) { return CROSS ? k_used : k_used + t; };
      auto v_idx = [&](int t) { return CROSS ? v_used : v_used + t; };
      auto q_idx = [&](int t) { return CROSS ? qd_used + t : qd_used; };
      auto q_base = [&](int t) { return sQD + (q_idx(t) % C::kQDStages) * 2 * kChunkBytes; };
      // S^T = K Q^T and dP^T = V dO^T of step t, once its tiles have landed. They
      // overwrite the P^T / dS^T columns of the step before, which the dV / dK
      // products issued before them have read (in order).
      auto issue_sdp = [&](int t) -> bool {
        const uint32_t ki = k_idx(t), vi = v_idx(t), qi = q_idx(t);
        const int ks = ki % C::kKStages, vs = vi % C::kVStages, qs = qi % C::kQDStages;
        if ((CROSS || t == 0) && !wait_bar(&bars->qd_full[qs], (qi / C::kQDStages) & 1, abort_flag, a, 97))
          return false;
        if ((!CROSS || t == 0) && !wait_bar(&bars->k_full[ks], (ki / C::kKStages) & 1, abort_flag, a, 98))
          return false;
        tc_fence_after();
        const uint64_t dQk = sdesc_sw128(q_base(t), 16, 1024), dDOk = sdesc_sw128(q_base(t) + kChunkBytes, 16, 1024);
        const uint64_t kd = dK0 + ks * (kTileBytes >> 4), vd = dV0 + vs * (kTileBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem + C::kSCol, kd + kslice(kk, kBoxK), dQk + kslice(kk, kBoxQ), idS, kk > 0 ? 1u : 0u);
        mma_commit(&bars->s_full);
        if (!CROSS || t == 0) {
          if (!wait_bar(&bars->v_full[vs], (vi / C::kVStages) & 1, abort_flag, a, 99)) return false;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(tmem + C::kDPCol, vd + kslice(kk, kBoxK), dDOk + kslice(kk, kBoxQ), idS, kk > 0 ? 1u : 0u);
        mma_commit(&bars->dp_full);
        if constexpr (!CROSS) mma_commit(&bars->v_empty[vs]);
        return true;
      };
      for (long long r = 0; ok && load_bitem<CROSS>(a, r, it); ++r) {
        if (it.hi <= it.lo) continue;
        const int ns = it.hi - it.lo;
        if (!(ok = issue_sdp(0))) break;
        for (int t = 0; t < ns; ++t) {
          const uint32_t nt = n + t;
          const int ks = k_idx(t) % C::kKStages, qs = q_idx(t) % C::kQDStages;
          const uint64_t dQm = sdesc_sw128(q_base(t), kBoxQ, 1024), dDOm = sdesc_sw128(q_base(t) + kChunkBytes, kBoxQ, 1024);
          const uint64_t ktd = dKt0 + ks * (kTileBytes >> 4);
          // dV = P^T dO once P^T is in TMEM and the epilogue has drained the
          // accumulators of the group before (pooling: each step; cross: each item)
          const bool acc_first = CROSS ? t == 0 : true;
          if (!(ok = wait_bar(&bars->p_ready, nt & 1, abort_flag, a, 100))) break;
          if (acc_first && !(ok = wait_bar(&bars->acc_empty, (acc_n & 1) ^ 1, abort_flag, a, 101))) break;
          tc_fence_after();
#pragma unroll
          for (int hl = 0; hl < C::kNP; ++hl)
#pragma unroll
            for (int kk = 0; kk < kQC / 16; ++kk)
              mma_ts(tmem + C::kDVCol, tmem + C::kSCol + 16 * hl + a_col(kk), dDOm + mnslice(kk), idG,
                     (!acc_first || hl > 0 || kk > 0) ? 1u : 0u);
          if (!(ok = wait_bar(&bars->ds_ready, nt & 1, abort_flag, a, 102))) break;
          tc_fence_after();
#pragma unroll
          for (int hl = 0; hl < C::kNP; ++hl)
#pragma unroll
            for (int kk = 0; kk < kQC / 16; ++kk)
              mma_ts(tmem + C::kDKCol, tmem + C::kDPCol + 16 * hl + a_col(kk), dQm + mnslice(kk), idG,
                     (!acc_first || hl > 0 || kk > 0) ? 1u : 0u);
          if constexpr (!CROSS) {
            mma_commit(&bars->acc_full);
            ++acc_n;
          }
          // the next step's S^T and dP^T go ahead of this step's dQ^T, so the
          // activation of the next step overlaps it
          if (t + 1 < ns && !(ok = issue_sdp(t + 1))) break;
          // dQ^T += K^T dS^T (pooling: over the item's steps; cross: one step)
          const bool dq_first = CROSS ? true : t == 0;
          if (dq_first && !(ok = wait_bar(&bars->dq_empty, (dq_n & 1) ^ 1, abort_flag, a, 103))) break;
#pragma unroll
          for (int hl = 0; hl < C::kNP; ++hl)
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ss(tmem + C::kDQCol, ktd + mnslice(kk), dDS0 + hl * (kPBytes >> 4) + mnslice(kk), idQ,
                     (!dq_first || hl > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bars->dsm_free);
          if constexpr (CROSS) {
            mma_commit(&bars->qd_empty[qs]);
            mma_commit(&bars->dq_full);
            ++dq_n;
          } else {
            mma_commit(&bars->k_empty[ks]);
          }
        }
        if (!ok) break;
        if constexpr (CROSS) {
          mma_commit(&bars->acc_full);
          ++acc_n;
          mma_commit(&bars->k_empty[0]);
          mma_commit(&bars->v_empty[0]);
          ++k_used;
          ++v_used;
          qd_used += ns;
        } else {
          mma_commit(&bars->qd_empty[qd_used % C::kQDStages]);
          mma_commit(&bars->dq_full);
          ++dq_n;
          ++qd_used;
          k_used += ns;
          v_used += ns;
        }
        n += ns;
      }
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, a.timeout_ns);
    }
    __syncwarp();
  }
  } else if (warp < 12) {
    // ------------------------------------------------------------ activation warpgroups
    // warpgroup g takes query columns [32 g, 32 g + 32) of every step (the
    // launch's register count is its share)
    const int g = (warp - 4) >> 2;
    const int row = 32 * (warp & 3) + lane;  // key row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_base + C::kSCol + 32 * g, tDP = tmem + lane_base + C::kDPCol + 32 * g;
    const uint32_t sDS = smem_u32(sm + C::kDSOff);
    uint32_t n = 0;
    bool ok = true;
    PItem it;
    for (long long r = 0; ok && load_bitem<CROSS>(a, r, it); ++r) {
      if (it.hi <= it.lo) continue;
      const int ns = it.hi - it.lo;
      for (int t = 0; t < ns; ++t) {
        const uint32_t nt = n + t;
        // key rows past the sequence and query columns past the chunk are
        // zero in P^T and dS^T: dV and dK sum over the query columns, dQ^T
        // over the key rows
        const int j = CROSS ? it.rt : it.lo + t;
        const bool valid = j * kTile + row < it.lkv;
        const int nq = (CROSS ? min(kQC, it.lq - (it.lo + t) * kQC) : it.lq) - 32 * g;  // this group's columns
        const bool any = nq > 0;
        ok = __all_sync(0xffffffffu, wait_bar(&bars->s_full, nt & 1, abort_flag, a, 104));
        if (!ok) break;
        tc_fence_after();
        uint32_t s[32];
        float gr[32];  // act'(x) of the group's query columns
        if (any) {
          tmem_ld32(tS, s);
          tmem_ld_wait();
        }
        // P^T as bf16: hi parts over the group's first 16 columns, lo parts the next 16
        uint32_t hi[16], lo[16];
        if (any) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int q = 2 * e;
            float f0, f1, g0, g1;
            act_and_grad<ACT>(__uint_as_float(s[q]) * a.scale, f0, g0);
            act_and_grad<ACT>(__uint_as_float(s[q + 1]) * a.scale, f1, g1);
            const bool a0 = valid && q < nq, a1 = valid && q + 1 < nq;
            f0 = a0 ? f0 : 0.0f;
            f1 = a1 ? f1 : 0.0f;
            gr[q] = a0 ? g0 : 0.0f;
            gr[q + 1] = a1 ? g1 : 0.0f;
            hi[e] = pack_bf16x2(f0, f1);
            if constexpr (HILO) lo[e] = bf16x2_lo(f0, f1, hi[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) hi[e] = lo[e] = 0u;
        }
        tmem_st16(tS, hi);
        if constexpr (HILO) tmem_st16(tS + 16, lo);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_ready);

        ok = __all_sync(0xffffffffu, wait_bar(&bars->dp_full, nt & 1, abort_flag, a, 105));
        if (!ok) break;
        tc_fence_after();
        if (any) {
          tmem_ld32(tDP, s);
          tmem_ld_wait();
        }
        // the dQ^T products of the step before have read the shared dS^T tile
        ok = __all_sync(0xffffffffu, wait_bar(&bars->dsm_free, (nt & 1) ^ 1, abort_flag, a, 106));
        if (!ok) break;
        if (any) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int q = 2 * e;
            const float d0 = gr[q] * __uint_as_float(s[q]), d1 = gr[q + 1] * __uint_as_float(s[q + 1]);
            hi[e] = pack_bf16x2(d0, d1);
            if constexpr (HILO) lo[e] = bf16x2_lo(d0, d1, hi[e]);
          }
        }
        tmem_st16(tDP, hi);
        if constexpr (HILO) tmem_st16(tDP + 16, lo);
        st_pt_row(sDS, row, 32 * g, hi);
        if constexpr (HILO) st_pt_row(sDS + kPBytes, row, 32 * g, lo);
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->ds_ready);
      }
      if (!ok) break;
      n += ns;
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
    // ------------------------------------------------------------ epilogue warpgroup
    // dV and dK rows (thread = key row) after each accumulation group, dQ
    // rows (thread = head-dim row) from dQ^T after each of its groups. Items
    // without keys (pooling) get zero dQ rows; items without queries (cross)
    // zero dK and dV rows.
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    uint32_t acc_n = 0, dq_n = 0;
    PItem it;
    bool ok = true;
    auto drain_kv = [&](int j, float cn) -> bool {
      if (!__all_sync(0xffffffffu, wait_bar(&bars->acc_full, acc_n & 1, abort_flag, a, 107))) return false;
      ++acc_n;
      tc_fence_after();
      const int jl = j * kTile + row;
      const bool valid = jl < it.lkv;
      const int64_t gk = it.k0 + jl;
      __nv_bfloat16* dv_row = a.out1 + (gk * a.H + it.h) * kD;
      __nv_bfloat16* dk_row = a.out2 + (gk * a.H + it.h) * kD;
#pragma unroll 1
      for (int c = 0; c < 2 * kD / 32; ++c) {
        const bool is_dk = c >= kD / 32;
        const int cc = is_dk ? c - kD / 32 : c;
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + (is_dk ? C::kDKCol : C::kDVCol) + 32 * cc, v);
        tmem_ld_wait();
        if (c == 2 * kD / 32 - 1) {
          tc_fence_before();
          mbar_arrive(&bars->acc_empty);
        }
        if (valid) {
          uint32_t w[16];
          const float mul = is_dk ? cn * a.scale : cn;
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
          store_words16((is_dk ? dk_row : dv_row) + 32 * cc, w, a.out_v8);
        }
      }
      return true;
    };
    auto drain_q = [&](int64_t q_first, int nq, float mul) -> bool {
      if (!__all_sync(0xffffffffu, wait_bar(&bars->dq_full, dq_n & 1, abort_flag, a, 108))) return false;
      ++dq_n;
      tc_fence_after();
      const int halves = nq > 32 ? 2 : 1;
#pragma unroll 1
      for (int c = 0; c < halves; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + C::kDQCol + 32 * c, v);
        tmem_ld_wait();
        if (c == halves - 1) {  // dQ^T is free for the next group once read
          tc_fence_before();
          mbar_arrive(&bars->dq_empty);
        }
        store_chunk_cols(a.out0, q_first, nq, a.H, it.h, row, 32 * c, v, mul);
      }
      return true;
    };
    for (long long r = 0; ok && load_bitem<CROSS>(a, r, it); ++r) {
      if (it.hi <= it.lo) {
        if constexpr (CROSS) {
          const int jl = it.rt * kTile + row;
          if (jl < it.lkv) {
            const int64_t gk = it.k0 + jl;
            uint4* dv = reinterpret_cast<uint4*>(a.out1 + (gk * a.H + it.h) * kD);
            uint4* dk = reinterpret_cast<uint4*>(a.out2 + (gk * a.H + it.h) * kD);
            for (int e = 0; e < kD / 8; ++e) dv[e] = dk[e] = make_uint4(0, 0, 0, 0);
          }
        } else {
          store_chunk_cols(a.out0, it.q0, it.lq, a.H, it.h, row, 0, nullptr, 0.0f);
          store_chunk_cols(a.out0, it.q0, it.lq, a.H, it.h, row, 32, nullptr, 0.0f);
        }
        continue;
      }
      const int ns = it.hi - it.lo;
      const float cn = (a.norm_by_lkv && it.lkv > 0) ? 1.0f / it.lkv : 1.0f;
      for (int t = 0; t < ns && ok; ++t) {
        if constexpr (CROSS) {
          const int c = it.lo + t;
          ok = drain_q(it.q0 + static_cast<int64_t>(c) * kQC, min(kQC, it.lq - c * kQC), cn * a.scale);
        } else {
          ok = drain_kv(it.lo + t, cn);
        }
      }
      if (!ok) break;
      ok = CROSS ? drain_kv(it.rt, cn) : drain_q(it.q0, it.lq, cn * a.scale);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// Whether every sequence suits the fused backward's mode. Pooling: 1 <= Lq
// <= 64, or no keys. Cross: Lkv <= 128, and keys whenever there are queries.
// If so, the general dQ and dK/dV schedules are emptied so their passes find
// no work; else the gate stays closed and the fused pass returns.
__global__ void __launch_bounds__(1024) pma_gate_kernel(const int64_t* q_off, const int64_t* kv_off, int64_t B,
                                                        int cross, int* gate, int* n_tiles_q, int* n_tiles_kv) {
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int64_t b = threadIdx.x; b < B; b += blockDim.x) {
    const int64_t lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
    bool ok = lq >= 0 && lkv >= 0;
    if (cross) ok = ok && lkv <= kTile && (lkv > 0 || lq == 0);
    else ok = ok && lq <= kQC && (lq > 0 || lkv == 0);
    if (!ok) bad = 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    *gate = bad ? 0 : 1;
    if (!bad) {
      *n_tiles_q = 0;
      *n_tiles_kv = 0;
    }
  }
}

template <typename K>
cudaError_t launch_k(K kernel, int smem, int grid, cudaStream_t st, const CUtensorMap& q, const CUtensorMap& k,
                     const CUtensorMap& v, const AttnArgs& a) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, smem, st>>>(q, k, v, a);
  return cudaGetLastError();
}

template <int ACT>
cudaError_t fwd_act(bool hilo, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const AttnArgs& a,
                    int grid, cudaStream_t st) {
  if (hilo) return launch_k(pma_fwd_kernel<ACT, true>, PfCfg<true>::kSmemBytes, grid, st, q, k, v, a);
  return launch_k(pma_fwd_kernel<ACT, false>, PfCfg<false>::kSmemBytes, grid, st, q, k, v, a);
}

template <int ACT, bool HILO, bool CROSS>
cudaError_t bwd_one(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                    const AttnArgs& a, const int* gate, int grid, cudaStream_t st) {
  auto kernel = pma_bwd_kernel<ACT, HILO, CROSS>;
  constexpr int smem = PbCfg<HILO, CROSS>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kBwdThreads, smem, st>>>(q, k, v, dout, a, gate);
  return cudaGetLastError();
}

template <int ACT>
cudaError_t bwd_act(bool hilo, bool cross, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                    const CUtensorMap& dout, const AttnArgs& a, const int* gate, int grid, cudaStream_t st) {
  if (cross)
    return hilo ? bwd_one<ACT, true, true>(q, k, v, dout, a, gate, grid, st)
                : bwd_one<ACT, false, true>(q, k, v, dout, a, gate, grid, st);
  return hilo ? bwd_one<ACT, true, false>(q, k, v, dout, a, gate, grid, st)
              : bwd_one<ACT, false, false>(q, k, v, dout, a, gate, grid, st);
}

template <int ACT>
cudaError_t skv_act(bool hilo, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const AttnArgs& a,
                    const int* gate, int grid, cudaStream_t st) {
  auto kernel = hilo ? skv_fwd_kernel<ACT, true> : skv_fwd_kernel<ACT, false>;
  constexpr int smem = SfCfg<false>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, smem, st>>>(q, k, v, a, gate);
  return cudaGetLastError();
}

template <int ACT>
cudaError_t skvb_act(bool hilo, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                     const CUtensorMap& dout, const AttnArgs& a, const int* gate, int grid, cudaStream_t st) {
  auto kernel = hilo ? skv_bwd_kernel<ACT, true> : skv_bwd_kernel<ACT, false>;
  const int smem = hilo ? SbCfg<true>::kSmemBytes : SbCfg<false>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kBwdThreads, smem, st>>>(q, k, v, dout, a, gate);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_skv_bwd(int act, bool hilo, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& dout, const AttnArgs& a, const int* gate, int grid,
                           cudaStream_t stream) {
  switch (act) {
    case JATTN_SILU: return skvb_act<JATTN_SILU>(hilo, q, k, v, dout, a, gate, grid, stream);
    case JATTN_GELU_TANH: return skvb_act<JATTN_GELU_TANH>(hilo, q, k, v, dout, a, gate, grid, stream);
    case JATTN_GELU_POLY: return skvb_act<JATTN_GELU_POLY>(hilo, q, k, v, dout, a, gate, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_pma_fwd(int act, bool hilo, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const AttnArgs& a, int grid, cudaStream_t stream) {
  switch (act) {
    case JATTN_SILU: return fwd_act<JATTN_SILU>(hilo, q, k, v, a, grid, stream);
    case JATTN_GELU_TANH: return fwd_act<JATTN_GELU_TANH>(hilo, q, k, v, a, grid, stream);
    case JATTN_GELU_POLY: return fwd_act<JATTN_GELU_POLY>(hilo, q, k, v, a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_skv_fwd(int act, bool hilo, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const AttnArgs& a, const int* gate, int grid, cudaStream_t stream) {
  switch (act) {
    case JATTN_SILU: return skv_act<JATTN_SILU>(hilo, q, k, v, a, gate, grid, stream);
    case JATTN_GELU_TANH: return skv_act<JATTN_GELU_TANH>(hilo, q, k, v, a, gate, grid, stream);
    case JATTN_GELU_POLY: return skv_act<JATTN_GELU_POLY>(hilo, q, k, v, a, gate, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_pma_gate(const int64_t* q_off, const int64_t* kv_off, int64_t B, bool cross, int* gate,
                            int* n_tiles_q, int* n_tiles_kv, cudaStream_t stream) {
  pma_gate_kernel<<<1, 1024, 0, stream>>>(q_off, kv_off, B, cross ? 1 : 0, gate, n_tiles_q, n_tiles_kv);
  return cudaGetLastError();
}

cudaError_t launch_pma_bwd(int act, bool hilo, bool cross, const CUtensorMap& q, const CUtensorMap& k,
                           const CUtensorMap& v, const CUtensorMap& dout, const AttnArgs& a, const int* gate,
                           int grid, cudaStream_t stream) {
  switch (act) {
    case JATTN_SILU: return bwd_act<JATTN_SILU>(hilo, cross, q, k, v, dout, a, gate, grid, stream);
    case JATTN_GELU_TANH: return bwd_act<JATTN_GELU_TANH>(hilo, cross, q, k, v, dout, a, gate, grid, stream);
    case JATTN_GELU_POLY: return bwd_act<JATTN_GELU_POLY>(hilo, cross, q, k, v, dout, a, gate, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int pma_rows_per_item() { return kQC; }

}  // namespace jattn
