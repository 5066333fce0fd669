// Host-side launchers of the attention kernels.
#pragma once
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace jattn {

struct AttnArgs;
struct DevStatus;

// Forward: schedule rows are blocks of fwd_rows_per_item() query rows. `split`
// selects the column-split arrangement of the activation warps (for items that
// mostly hold one query tile) over the ping-pong one; `block` selects the
// kernels compiled for block masks (fwd_block.cu) and `hilo` those that pass P
// as bf16 hi + lo parts (pointwise activations without the 1/Lkv normaliser,
// fwd_hilo.cu, fwd_block_hilo.cu).
cudaError_t launch_fwd(int D, int act, bool split, bool block, bool hilo, const CUtensorMap& q, const CUtensorMap& k,
                       const CUtensorMap& v, const AttnArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_fwd_block(int D, int act, bool split, const CUtensorMap& q, const CUtensorMap& k,
                             const CUtensorMap& v, const AttnArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_fwd_hilo(int D, int act, bool split, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, const AttnArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_fwd_block_hilo(int D, int act, bool split, const CUtensorMap& q, const CUtensorMap& k,
                                  const CUtensorMap& v, const AttnArgs& a, int grid, cudaStream_t stream);
int fwd_rows_per_item();

// MXFP8 forward (softmax, D = 128): maps of the E4M3 codes (uint8 [rows, H*128],
// boxes of 128 rows x 128 bytes); a.sf_* / a.bs_* carry the block scales.
cudaError_t launch_fwd_mx(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const AttnArgs& a,
                          int grid, cudaStream_t stream);

// MXFP8 backward (softmax, D = 128). launch_mx_di: D_i = <dO~_i, O_i> per
// query row and head into di (row blocks from block_start, at most
// max_blocks of them). dq: over 128-row query tiles (maps of 128-row boxes);
// dkdv: over 128-row key tiles, queries in steps of 96 (the Q and dO maps
// have 96-row boxes). a.f0 = LSE, a.f1 = D; a.sf_* / a.bs_* the block scales.
cudaError_t launch_mx_di(const int64_t* q_off, int B, int H, int64_t max_blocks, const uint8_t* dout,
                         const uint8_t* dout_scales, const int* block_start, const void* o, float* di,
                         cudaStream_t stream);
cudaError_t launch_bwd_dq_mx(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const CUtensorMap& dout, const AttnArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_bwd_dkdv_mx(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& dout, const AttnArgs& a, int grid, cudaStream_t stream);

// dK, dV over key tiles (transposed schedule, 128-row key tiles); a.out0 /
// a.out1 receive dK / dV.
cudaError_t launch_bwd_dkdv(int D, int act, bool hilo, const CUtensorMap& q, const CUtensorMap& k,
                            const CUtensorMap& v, const CUtensorMap& dout, const AttnArgs& a, int grid,
                            cudaStream_t stream);
cudaError_t launch_bwd_dkdv_hilo(int D, int act, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& dout, const AttnArgs& a, int grid, cudaStream_t stream);
// dQ over query tiles (128-row query tiles). For softmax it also computes
// Di = rowsum(dO * O) from the dO tiles and O (the map `o` in the one-ring
// layout, the rows at a.in0 in the two-ring one) into a.f1, so it runs before
// the dK/dV pass, which reads Di. `split`: K and V tiles in two rings (used at
// D = 128, for items of many key tiles).
cudaError_t launch_bwd_dq(int D, int act, bool hilo, bool split, const CUtensorMap& q, const CUtensorMap& k,
                          const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& o, const AttnArgs& a,
                          int grid, cudaStream_t stream);
cudaError_t launch_bwd_dq_hilo(int D, int act, bool split, const CUtensorMap& q, const CUtensorMap& k,
                               const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& o, const AttnArgs& a,
                               int grid, cudaStream_t stream);

// Short-query / short-key attention (pma.cu): pointwise activations, no
// mask, D = 128, keys on the MMA's M dimension and at most 64 queries per
// product. The forward takes items of at most 64 query rows from the 64-row
// query-tile schedule; its Q map has 64-row boxes (a.out0 = O). The fused
// backward (Q and dO maps with 64-row boxes; a.out0 = dQ, a.out1 = dV, a.out2
// = dK) has a pooling mode (items from the 64-row query-tile schedule, every
// sequence with 1 <= Lq <= 64 or no keys) and a cross mode (`cross`: items
// from the 128-row key-tile schedule with 64-column query ranges, every
// sequence with Lkv <= 128 and keys whenever it has queries). It runs only
// when launch_pma_gate found the batch within its mode's limits; the gate
// then empties the general dQ and dK/dV schedules.
cudaError_t launch_pma_fwd(int act, bool hilo, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const AttnArgs& a, int grid, cudaStream_t stream);
// Short-key forward (pma.cu): cross-attention whose every sequence has at
// most 128 keys (the gate's cross mode), items from the 128-row key-tile
// schedule with 128-row query ranges; Q map with 128-row boxes, a.out0 = O.
cudaError_t launch_skv_fwd(int act, bool hilo, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const AttnArgs& a, const int* gate, int grid, cudaStream_t stream);
// Short-key backward (pma.cu): the same shapes and schedule as
// launch_skv_fwd (128-row query ranges), Q / dO maps with 128-row boxes;
// a.out0 = dQ, a.out1 = dV, a.out2 = dK.
cudaError_t launch_skv_bwd(int act, bool hilo, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& dout, const AttnArgs& a, const int* gate, int grid,
                           cudaStream_t stream);
cudaError_t launch_pma_gate(const int64_t* q_off, const int64_t* kv_off, int64_t B, bool cross, int* gate,
                            int* n_tiles_q, int* n_tiles_kv, cudaStream_t stream);
cudaError_t launch_pma_bwd(int act, bool hilo, bool cross, const CUtensorMap& q, const CUtensorMap& k,
                           const CUtensorMap& v, const CUtensorMap& dout, const AttnArgs& a, const int* gate,
                           int grid, cudaStream_t stream);
int pma_rows_per_item();

// Rotary embedding of a jagged tensor x ([total, H, D] bf16, rows described
// by own_off; other_off describes the other side for the alignment):
// y = R(pos) x, or R(pos)^T x with `inverse`. keys: x holds key rows.
cudaError_t launch_rope(const int64_t* own_off, const int64_t* other_off, int B, int keys, int inverse, int H,
                        int D, int64_t total, const void* x, void* y, const float* cos_t, const float* sin_t,
                        int rows, DevStatus* status, cudaStream_t stream);
// MXFP8 (E4M3 + one E8M0 scale per 32 x 32 block) quantization of a jagged
// bf16 tensor; block_start / n_blocks come from sched_prefix_launch(32).
cudaError_t launch_mx_quant(const int64_t* off, int B, int H, int D, int64_t max_blocks, const void* x, void* codes,
                            uint8_t* scales, const int* block_start, const int* n_blocks, cudaStream_t stream);
// Row-major [rows, half] cos / sin tables to pair-major [half, rows] copies.
cudaError_t launch_rope_transpose(const float* cos_t, const float* sin_t, int rows, int half, float* cos_pm,
                                  float* sin_pm, cudaStream_t stream);

}  // namespace jattn
