// Host interface of the device-side tile scheduler.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace jattn {

struct DevStatus;

// Views into one schedule's slice of the workspace.
struct SchedView {
  int* tile_start;  // [B+1] exclusive prefix of row tiles per sequence
  int* n_tiles;     // [1] number of row tiles
  int4* tmp;        // [max_tiles] tiles in (b, row tile) order
  int* hist;        // [nblk][1024] per-block cost counts, then output positions
  int4* sorted;     // [max_tiles] longest-first schedule
  int64_t max_tiles;
  int nblk;
};

int64_t sched_max_tiles(int64_t B, int64_t rows_total, int row_tile);
size_t sched_ws_bytes(int64_t B, int64_t max_tiles);
SchedView sched_carve(void* base, int64_t B, int64_t max_tiles);
// Only the checked offsets' prefix of ceil(L_b / row_tile) (no sort).
cudaError_t sched_prefix_launch(const int64_t* off, int64_t B, int64_t total, int row_tile, int* tile_start,
                                int* n_tiles, DevStatus* status, cudaStream_t stream);
cudaError_t sched_launch(const SchedView& v, const int64_t* q_off, const int64_t* kv_off, int64_t B,
                         int64_t total_q, int64_t total_kv, int row_tile, int col_tile, int mask, int window,
                         int transposed, DevStatus* status, cudaStream_t stream);

}  // namespace jattn
