// Device-side tile scheduler.
//
// "GEM Training" post, GDPA section, bullet on software tile scheduling for
// jagged tensors: valid tiles are enumerated up front, empty ones are never
// launched, and the rest are spread across the SMs so that no SM receives a
// much longer share. Here the enumeration runs on the device from the offsets
// (no host round trip), and the order is longest-first: a stable counting
// sort by the number of column tiles a row tile must visit, ties in
// (sequence, row tile) order. The persistent kernels then deal the sorted
// list out zigzag across their CTAs.
#include <cstdint>

#include "common.cuh"
#include "sched.h"

namespace jattn {

namespace {

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  total = warp_sums[nwarps - 1];
  __syncthreads();
  return before;
}

// Validate offsets, count row tiles per sequence and prefix-sum them.
__global__ void __launch_bounds__(1024) sched_prep(const int64_t* __restrict__ q_off,
                                                   const int64_t* __restrict__ kv_off, int64_t B,
                                                   int64_t total_q, int64_t total_kv, int row_tile,
                                                   int transposed, int* __restrict__ tile_start,
                                                   int* __restrict__ n_tiles, DevStatus* status) {
  __shared__ int warp_sums[32];
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    if (q_off[0] != 0 || kv_off[0] != 0 || q_off[B] != total_q || kv_off[B] != total_kv) {
      bad = 1;
      record_error(status, JATTN_ERR_OFFSETS, 1, -1);
    }
  }
  for (int64_t b = threadIdx.x; b < B; b += blockDim.x) {
    if (q_off[b + 1] < q_off[b] || kv_off[b + 1] < kv_off[b]) {
      bad = 1;
      record_error(status, JATTN_ERR_OFFSETS, 2, static_cast<int>(b));
    }
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) *n_tiles = 0;
    return;
  }
  int carry = 0;
  for (int64_t base = 0; base < B; base += blockDim.x) {
    const int64_t b = base + threadIdx.x;
    int n = 0;
    if (b < B) {
      const int64_t rows = transposed ? (kv_off[b + 1] - kv_off[b]) : (q_off[b + 1] - q_off[b]);
      n = static_cast<int>((rows + row_tile - 1) / row_tile);
    }
    int total;
    const int ex = block_exclusive_scan(n, warp_sums, total);
    if (b < B) tile_start[b] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) {
    tile_start[B] = carry;
    *n_tiles = carry;
  }
}

__global__ void __launch_bounds__(kSchedBlock) sched_hist(const int64_t* __restrict__ q_off,
                                                          const int64_t* __restrict__ kv_off, int64_t B,
                                                          const int* __restrict__ tile_start,
                                                          const int* __restrict__ n_tiles, int row_tile,
                                                          int col_tile, int mask, int window, int transposed,
                                                          int4* __restrict__ tmp, int* __restrict__ hist) {
  __shared__ int h[kCostBuckets];
  for (int i = threadIdx.x; i < kCostBuckets; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int T = *n_tiles;
  const int t = blockIdx.x * kSchedBlock + threadIdx.x;
  if (t < T) {
    // b = (last index with tile_start[b] <= t) among 0..B
    int64_t lo = 0, hi = B;  // invariant: tile_start[lo] <= t < tile_start[hi + ...]
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) >> 1;
      if (tile_start[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    const int b = static_cast<int>(lo);
    const int rt = t - tile_start[b];
    const int lq = static_cast<int>(q_off[b + 1] - q_off[b]);
    const int lkv = static_cast<int>(kv_off[b + 1] - kv_off[b]);
    int c_lo, c_hi;
    tile_range(lq, lkv, rt, row_tile, col_tile, mask, window, transposed, c_lo, c_hi);
    tmp[t] = make_int4(b, rt, c_lo, c_hi);
    atomicAdd(&h[min(c_hi - c_lo, kCostBuckets - 1)], 1);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kCostBuckets; i += blockDim.x) hist[blockIdx.x * kCostBuckets + i] = h[i];
}

// Turn per-block bucket counts into global output positions: descending cost,
// and within a cost, block order (= tile order).
__global__ void __launch_bounds__(kCostBuckets) sched_scan(int* __restrict__ hist, int nblk) {
  __shared__ int warp_sums[32];
  __shared__ int start[kCostBuckets];
  const int c = threadIdx.x;
  int running = 0;
  for (int blk = 0; blk < nblk; ++blk) {
    const int x = hist[blk * kCostBuckets + c];
    hist[blk * kCostBuckets + c] = running;
    running += x;
  }
  // exclusive scan over buckets from the most expensive down
  const int rc = kCostBuckets - 1 - c;
  __shared__ int totals[kCostBuckets];
  totals[c] = running;
  __syncthreads();
  int total;
  const int ex = block_exclusive_scan(totals[rc], warp_sums, total);
  start[rc] = ex;
  __syncthreads();
  const int s = start[c];
  for (int blk = 0; blk < nblk; ++blk) hist[blk * kCostBuckets + c] += s;
}

__global__ void __launch_bounds__(kSchedBlock) sched_place(const int4* __restrict__ tmp,
                                                           const int* __restrict__ hist,
                                                           const int* __restrict__ n_tiles,
                                                           int4* __restrict__ sorted) {
  __shared__ int base[kCostBuckets];
  for (int i = threadIdx.x; i < kCostBuckets; i += blockDim.x) base[i] = hist[blockIdx.x * kCostBuckets + i];
  const int T = *n_tiles;
  const int t = blockIdx.x * kSchedBlock + threadIdx.x;
  const bool valid = t < T;
  int4 tile = make_int4(0, 0, 0, 0);
  int c = 0;
  if (valid) {
    tile = tmp[t];
    c = min(tile.w - tile.z, kCostBuckets - 1);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned key = valid ? static_cast<unsigned>(c) : static_cast<unsigned>(kCostBuckets + lane);
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  const int leader = __ffs(peers) - 1;
  int pos = 0;
  for (int w = 0; w < kSchedBlock / 32; ++w) {
    __syncthreads();
    if (warp == w) {
      if (valid) pos = base[c] + rank;
      __syncwarp();
      if (valid && lane == leader) base[c] += __popc(peers);
    }
  }
  if (valid) sorted[pos] = tile;
}

}  // namespace

int64_t sched_max_tiles(int64_t B, int64_t rows_total, int row_tile) {
  return rows_total / row_tile + B + 1;
}

size_t sched_ws_bytes(int64_t B, int64_t max_tiles) {
  const int64_t nblk = (max_tiles + kSchedBlock - 1) / kSchedBlock;
  size_t n = 0;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  n += al(sizeof(int) * (B + 1));          // tile_start
  n += al(sizeof(int) * 4);                // n_tiles
  n += al(sizeof(int4) * max_tiles);       // tmp
  n += al(sizeof(int) * nblk * kCostBuckets);  // hist
  n += al(sizeof(int4) * max_tiles);       // sorted
  return n;
}

SchedView sched_carve(void* base, int64_t B, int64_t max_tiles) {
  const int64_t nblk = (max_tiles + kSchedBlock - 1) / kSchedBlock;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  char* p = static_cast<char*>(base);
  SchedView v;
  v.tile_start = reinterpret_cast<int*>(p);
  p += al(sizeof(int) * (B + 1));
  v.n_tiles = reinterpret_cast<int*>(p);
  p += al(sizeof(int) * 4);
  v.tmp = reinterpret_cast<int4*>(p);
  p += al(sizeof(int4) * max_tiles);
  v.hist = reinterpret_cast<int*>(p);
  p += al(sizeof(int) * nblk * kCostBuckets);
  v.sorted = reinterpret_cast<int4*>(p);
  v.max_tiles = max_tiles;
  v.nblk = static_cast<int>(nblk);
  return v;
}

cudaError_t sched_prefix_launch(const int64_t* off, int64_t B, int64_t total, int row_tile, int* tile_start,
                                int* n_tiles, DevStatus* status, cudaStream_t stream) {
  sched_prep<<<1, 1024, 0, stream>>>(off, off, B, total, total, row_tile, 0, tile_start, n_tiles, status);
  return cudaGetLastError();
}

cudaError_t sched_launch(const SchedView& v, const int64_t* q_off, const int64_t* kv_off, int64_t B,
                         int64_t total_q, int64_t total_kv, int row_tile, int col_tile, int mask, int window,
                         int transposed, DevStatus* status, cudaStream_t stream) {
  sched_prep<<<1, 1024, 0, stream>>>(q_off, kv_off, B, total_q, total_kv, row_tile, transposed, v.tile_start,
                                     v.n_tiles, status);
  sched_hist<<<v.nblk, kSchedBlock, 0, stream>>>(q_off, kv_off, B, v.tile_start, v.n_tiles, row_tile, col_tile,
                                                 mask, window, transposed, v.tmp, v.hist);
  sched_scan<<<1, kCostBuckets, 0, stream>>>(v.hist, v.nblk);
  sched_place<<<v.nblk, kSchedBlock, 0, stream>>>(v.tmp, v.hist, v.n_tiles, v.sorted);
  return cudaGetLastError();
}

}  // namespace jattn
