/*
 * jattn: jagged generalized dot-product attention on one GB300 (sm_103a).
 *
 * The operation ("GEM Training" engineering post, section "Jagged Sequence
 * Flash Attention": attention computed directly on variable-length jagged
 * tensors, with asymmetric query and key/value lengths, without padding;
 * section "Generalized Dot-Product Attention (GDPA)": the same two matrix
 * products with an element-wise GELU or SiLU in place of the softmax, one
 * kernel for self-, cross- and pooling attention; section "BlockAttention":
 * sliding windows for long self-attention, then fixed blocks in which each
 * query block sees only its own key block). For every sequence b and head h,
 * with query rows i < Lq(b), key rows j < Lkv(b), delta = Lkv - Lq:
 *
 *   allowed(i, j)  causal: j <= i + delta;  window W: 0 <= i + delta - j < W;
 *                  block W: floor(j / W) == floor((i + delta) / W)
 *   s_ij = scale * <q_i, k_j>
 *   JATTN_SOFTMAX     o_i = sum_j softmax_j(s_ij) v_j over allowed j,
 *                     lse_i = ln sum_j exp(s_ij)  (no allowed key: o_i = 0,
 *                     lse_i = -inf)
 *   JATTN_SILU / JATTN_GELU_TANH / JATTN_GELU_POLY
 *                     o_i = c * sum_{allowed j} act(s_ij) v_j, c = 1/Lkv(b)
 *                     when norm_by_lkv, else 1
 *
 * and the backward pass gives dQ, dK, dV of a loss L from dO = dL/dO.
 *
 * Data layout. Jagged tensors are dense row-major [total, H, D] arrays of
 * bf16 (passed as uint16_t bit patterns) whose rows for sequence b are
 * off[b] .. off[b+1]-1; offsets are int64 [B+1] device arrays with off[0] = 0,
 * non-decreasing, off[B] = total. Self-attention passes the same offsets (and
 * may pass the same pointer) for queries and keys. lse is fp32 [total_q, H].
 * Every pointer argument except `p`, `bytes` and `device_status` is a DEVICE
 * pointer; value tensors must be 16-byte aligned.
 *
 * Ownership. The caller owns every buffer, including the workspace; the
 * library allocates no device memory, launches only on `stream` (a
 * cudaStream_t passed as void*, NULL = legacy default stream) and never
 * synchronises it in jattn_fwd / jattn_bwd. Calls are asynchronous: errors
 * that only the device can see (bad offsets, an expired bounded wait) are
 * written to a status word in the workspace and read by jattn_get_status.
 * Kernels never trap.
 *
 * Return codes: JATTN_OK or a JATTN_ERR_* value; jattn_error_string names it.
 */
#ifndef JATTN_H
#define JATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Activation between the two products. */
enum {
  JATTN_SOFTMAX = 0,   /* row softmax (Jagged Flash Attention) */
  JATTN_SILU = 1,      /* x / (1 + e^-x) (GDPA) */
  JATTN_GELU_TANH = 2, /* x/2 (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))) (GDPA) */
  /* GDPA's ALU-only GELU: the tanh-GELU above replaced by its Taylor
   * polynomial at 0 through x^6, evaluated with fused multiply-adds only
   * (section "Generalized Dot-Product Attention (GDPA)": no tanh on the
   * special-function unit, accurate on the score range that query/key
   * normalisation bounds). With c = sqrt(2/pi), a = 0.044715:
   *   act(x)  = x/2 + (c/2) x^2 + ((c a - c^3/3)/2) x^4 + ((2c^5/15 - c^3 a)/2) x^6
   *   act'(x) = its derivative (the backward differentiates the polynomial).
   * Within 1.2e-4 of tanh-GELU (derivative 1.3e-3) for |s| <= 0.75, and
   * 1.2e-3 (derivative 9e-3) for |s| <= 1; outside that range it departs
   * quickly (2.6e-2 at |s| = 1.5), so callers bound |s|, e.g. by normalising
   * query and key rows. */
  JATTN_GELU_POLY = 3
};

/* Mask bits. JATTN_MASK_WINDOW must be combined with JATTN_MASK_CAUSAL;
 * JATTN_MASK_BLOCK may be combined with JATTN_MASK_CAUSAL (causal inside each
 * block) but not with JATTN_MASK_WINDOW. Both read their width W from
 * jattn_params_t.window. */
enum { JATTN_MASK_NONE = 0, JATTN_MASK_CAUSAL = 1, JATTN_MASK_WINDOW = 2, JATTN_MASK_BLOCK = 4 };

enum {
  JATTN_OK = 0,
  JATTN_ERR_INVALID = 1,     /* bad argument detected on the host */
  JATTN_ERR_CUDA = 2,        /* a CUDA runtime call failed (launch, attribute) */
  JATTN_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned */
  JATTN_ERR_ALIGN = 4,       /* a value tensor is not 16-byte aligned */
  JATTN_ERR_OFFSETS = 5,     /* device: offsets not a valid prefix sum of the totals */
  JATTN_ERR_TIMEOUT = 6,     /* device: a bounded pipeline wait expired */
  JATTN_ERR_UNSUPPORTED = 7, /* device is not sm_103 / no kernel image */
  JATTN_ERR_TOO_LARGE = 8,   /* jattn_fwd_noalloc: problem needs more than the library's scratch */
  JATTN_ERR_ROPE = 9         /* device: a rotary position at or beyond the cos/sin tables' rows */
};

typedef struct {
  int64_t B;          /* number of sequences (1 .. 2^31 - 1) */
  int64_t total_q;    /* query rows = q_off[B] (>= 0) */
  int64_t total_kv;   /* key/value rows = kv_off[B] (>= 0) */
  int H;              /* heads (>= 1) */
  int D;              /* head dim: 64 or 128 */
  int act;            /* JATTN_SOFTMAX / JATTN_SILU / JATTN_GELU_TANH / JATTN_GELU_POLY */
  int mask;           /* JATTN_MASK_* bits: 0, CAUSAL, CAUSAL|WINDOW, BLOCK or CAUSAL|BLOCK */
  int window;         /* W >= 1: window width (WINDOW) or block size (BLOCK); else ignored */
  float scale;        /* > 0; 0 selects 1/sqrt(D) */
  int norm_by_lkv;    /* pointwise activations only: multiply by 1/Lkv(b) */
} jattn_params_t;

/* Precision. Products take bf16 operands with fp32 accumulation; P (and in
 * the backward dS) are rounded to bf16 before the second products, except
 * for pointwise activations with norm_by_lkv = 0: there every output sums
 * up to Lkv (or Lq) unscaled terms, so P and dS enter those products as two
 * bf16 parts, hi = bf16(x) and lo = bf16(x - hi), accumulating into the same
 * fp32 result (twice the tensor-core work of the second products). Results
 * then stay within |d| <= 1e-2 + 1e-2 |ref| of the exact attention at the
 * lengths tested (20000 keys per pooling query, 8000 queries per key). */

/* Bytes of workspace jattn_fwd / jattn_bwd need for these sizes (depends on
 * B, total_q, total_kv, H, D, act and mask only). The workspace must be 256-byte
 * aligned device memory whose first 256 bytes (the device status word) are
 * zero before its first use; jattn_get_status clears them again. Returns
 * JATTN_ERR_INVALID on bad params. */
int jattn_workspace_size(const jattn_params_t* p, size_t* bytes);

/* Pooling-shaped calls ("GEM Training" post, section "Generalized Dot-Product
 * Attention (GDPA)": a few learned queries per sequence against long key
 * sequences) run on kernels that put 128 keys on the MMA's M dimension
 * instead of a 128-row query tile that would be mostly padding: a pointwise
 * activation, mask JATTN_MASK_NONE, D = 128 and total_q <= 64 B. The forward
 * takes every such call (a sequence of more than 64 queries is served in
 * 64-row pieces). The backward fuses dQ, dK and dV into one pass over the
 * keys when every sequence has 1 <= Lq <= 64 or no keys. Cross-attention
 * over short key sequences (the same activation, mask and D, total_q > 64 B
 * and total_kv <= 128 B) runs a forward that keeps each sequence's one K/V
 * tile resident while its query tiles stream past, and a backward that fuses
 * the three gradients into one pass over 128-query tiles (dQ complete per
 * tile, dK and dV accumulated over the sequence), when every sequence has
 * Lkv <= 128, and keys whenever it has queries. These
 * conditions are checked on the device, without a host round trip; outside
 * them the general passes run. Results and their precision are the same as
 * on the general kernels. */

/* Forward. Reads q [total_q,H,D], k and v [total_kv,H,D]; writes every row of
 * o [total_q,H,D] and, for JATTN_SOFTMAX, lse [total_q,H] (must be non-NULL
 * then, except with JATTN_MASK_BLOCK, where NULL leaves LSE out; ignored for
 * pointwise activations). Host-side checks return JATTN_ERR_INVALID /
 * JATTN_ERR_ALIGN / JATTN_ERR_WORKSPACE without launching. Device-side
 * offset errors leave o unspecified and set the status word. */
int jattn_fwd(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint16_t* q,
              const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse, void* workspace,
              size_t workspace_bytes, void* stream);

/* Backward. Inputs as for jattn_fwd plus the forward's o and lse (softmax
 * only; ignored for pointwise activations) and dout [total_q,H,D]. Writes
 * every row of dq [total_q,H,D], dk and dv [total_kv,H,D]; key rows that no
 * query sees get zero gradients. The workspace may be the forward's.
 *
 * Softmax's D_i = <dO_i, O_i> is formed, for every 128-row query tile whose
 * allowed keys lie in one 128-row key tile, as sum_j P_ij dP_ij in fp32 from
 * that tile (exact, without the bf16 rounding of the stored O, which matters
 * for rows that see a few keys), and from o elsewhere.
 *
 * BlockAttention ("GEM Training" post, section "BlockAttention": blocks that
 * need no online softmax correction, no logsumexp traffic and no separate
 * D_i pass): with JATTN_MASK_BLOCK, a width that divides 128 (1, 2, 4, ...,
 * 128), softmax and self-attention passed as ONE offsets pointer (q_off ==
 * kv_off), every query tile meets exactly one key tile; the backward then
 * takes the row maximum, sum and D_i from that tile, reads neither o nor
 * lse (both may be NULL) and keeps the statistics it hands its dK/dV pass in
 * the workspace. */
int jattn_bwd(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint16_t* q,
              const uint16_t* k, const uint16_t* v, const uint16_t* o, const float* lse, const uint16_t* dout,
              uint16_t* dq, uint16_t* dk, uint16_t* dv, void* workspace, size_t workspace_bytes, void* stream);

/* Rotary position embedding (RoPE) around the attention ("GEM Training" post,
 * section "BlockAttention": the rotary backward fused into the attention
 * epilogue, so the gradients leave the kernel already rotated back, straight
 * from the fp32 accumulators, with no separate memory-bound pass).
 *
 * Rotation (the RoFormer form): dimensions pair up as (2m, 2m+1), m < D/2,
 * and R(pos) turns pair m by the angle pos * theta_m:
 *   y_2m   = x_2m cos - x_2m+1 sin,   y_2m+1 = x_2m sin + x_2m+1 cos,
 * with cos = rope_cos[pos * D/2 + m] and sin = rope_sin[pos * D/2 + m]: the
 * caller's fp32 device tables [rope_rows, D/2] (so theta, its base and any
 * scaling are the caller's), 16-byte aligned.
 * Positions: the queries and keys of a sequence end at the same position and
 * the longer side starts at 0 (the alignment of the masks):
 *   query row i -> i + max(delta, 0),  key row j -> j + max(-delta, 0),
 * delta = Lkv - Lq; every position must be < rope_rows (else the device
 * status becomes JATTN_ERR_ROPE and the affected rows are not rotated).
 *
 * jattn_rope: y = R(pos) x (inverse = 0) or R(pos)^T x (inverse = 1) for a
 * jagged tensor x of queries (keys = 0: [total_q,H,D]) or keys (keys = 1:
 * [total_kv,H,D]); y may alias x. A plain bandwidth-bound pass for the
 * forward side (the rotated q and k the forward reads). p supplies B, H, D
 * and the total of the rotated side (total_q or total_kv); both offset
 * arrays are read (the other side fixes the alignment). The workspace needs
 * only its first 256 bytes (the status word). Device pointers: q_off,
 * kv_off, x, y (16-byte aligned), rope_cos, rope_sin (16-byte aligned).
 *
 * Return codes (both rotary calls): JATTN_ERR_INVALID for bad params, a
 * missing table or rope_rows outside [1, INT32_MAX], keys / inverse not 0 or
 * 1; JATTN_ERR_ALIGN for misaligned tensors or tables; JATTN_ERR_WORKSPACE
 * for a workspace that is missing, misaligned or too small; JATTN_ERR_CUDA
 * when a launch fails. Nothing is launched when a host check fails.
 *
 * jattn_bwd_rope: jattn_bwd for attention on rotated queries and keys q' =
 * R q and k' = R k. It takes q' and k' (what the forward read) and returns
 * dq and dk with respect to the UNROTATED q and k: dq = R^T dL/dq',
 * dk = R^T dL/dk', applied in the dQ and dK epilogues. dv is unchanged.
 * Its workspace must hold jattn_bwd_rope_workspace_size bytes: the regular
 * layout plus pair-major copies of the tables ([D/2, rope_rows], made on
 * `stream` by the call), which let each warp of the epilogues read its 32
 * consecutive positions as one line. */
int jattn_bwd_rope_workspace_size(const jattn_params_t* p, int64_t rope_rows, size_t* bytes);
int jattn_rope(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, int keys, int inverse,
               const uint16_t* x, uint16_t* y, const float* rope_cos, const float* rope_sin, int64_t rope_rows,
               void* workspace, size_t workspace_bytes, void* stream);
int jattn_bwd_rope(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint16_t* q,
                   const uint16_t* k, const uint16_t* v, const uint16_t* o, const float* lse, const uint16_t* dout,
                   const float* rope_cos, const float* rope_sin, int64_t rope_rows, uint16_t* dq, uint16_t* dk,
                   uint16_t* dv, void* workspace, size_t workspace_bytes, void* stream);

/* MXFP8 quantization of a jagged tensor ("GEM Training" post, section "Low
 * Precision Flash Attention": block-scaled FP8 operands, FP8 data kept at the
 * unpadded positions with compact scales, and [32, 32] square blocks with one
 * scale each, so that a tensor quantized once serves both orientations).
 *
 * x: bf16 [total, H, D] rows described by off (int64 [B+1] device prefix
 * sums, checked like jattn_fwd's). codes: uint8 [total, H, D], the FP8 E4M3
 * code of every element at its own position. scales: uint8 E8M0 exponents
 * [jattn_mxfp8_scale_rows(B, total), H, D/32]; row block g of sequence b
 * (its sequence-local rows 32r .. 32r+31, the last block ragged) is
 * g = block_start[b] + r, and block_start (device int32 [B+1]) receives the
 * exclusive prefix sum of ceil(L_b / 32). For a block with largest magnitude
 * amax: E = max(0, floor(log2(amax)) - 8 + 127) (0 for an all-zero block),
 * X = 2^(E - 127), code = E4M3(x / X) rounded to nearest even and saturated
 * to +-448. Only the 32 * 32 block rows that exist are written. x and codes
 * 16-byte aligned; the workspace needs 512 bytes (status word + a count).
 * Bad offsets set JATTN_ERR_OFFSETS in the status word and write nothing.
 * Return codes: JATTN_ERR_INVALID (B < 1, totals or B beyond INT32_MAX,
 * H < 1, D not 64 / 128, a missing pointer), JATTN_ERR_ALIGN,
 * JATTN_ERR_WORKSPACE, JATTN_ERR_CUDA (launch failed); the caller owns every
 * buffer and scales has room for jattn_mxfp8_scale_rows(B, total) rows (an
 * upper bound: total/32 + B). */
int64_t jattn_mxfp8_scale_rows(int64_t B, int64_t total);
int jattn_mxfp8_quantize(int64_t B, int64_t total, int H, int D, const int64_t* off, const uint16_t* x,
                         uint8_t* codes, uint8_t* scales, int32_t* block_start, void* workspace,
                         size_t workspace_bytes, void* stream);

/* MXFP8 attention forward ("GEM Training" post, section "Low Precision Flash
 * Attention": FlashAttention on block-scaled FP8 operands, scale factors held
 * in tensor memory beside the accumulators, and the softmax output quantized
 * to FP8 inside the softmax with the scale its row maximum fixes).
 *
 * Softmax attention (p->act = JATTN_SOFTMAX, p->D = 128, norm_by_lkv = 0, any
 * mask of jattn_fwd) whose Q, K and V arrive as jattn_mxfp8_quantize output:
 * E4M3 codes [total, H, 128] (16-byte aligned) with E8M0 scales [row blocks,
 * H, 4] (4-byte aligned) and the row-block starts (int32 [B+1]) of their
 * offsets; K and V share kv_block_start (quantized with the same offsets).
 * Both products run as block-scaled tensor-core MMAs on the exact values the
 * codes and scales stand for, accumulating in fp32. P = exp(s - m), m the
 * running row maximum (moved when a row's maximum grows by more than 2^8), is
 * quantized per row and 32-key block with the scale 2^(ceil(log2 x) - 8), x
 * the block's largest P, so codes stay within E4M3's range and small values
 * keep their precision. The row sum l and LSE use the unquantized P in fp32;
 * o = (sum_j P~_ij v_j) / l (bf16), lse as jattn_fwd. Against quantizing with
 * the exact final maximum (the definition, scale 2^-8), each P~ differs by at
 * most one E4M3 rounding step (2^-3 P relative, below 2^-16 absolute in E4M3's
 * subnormal range), so |o - o_ref| <= sum_j (2^-3 p_ij + 2^-16 / l_i) |v_j|
 * plus the bf16 rounding of o. The workspace is jattn_fwd's (it uses the
 * 128-row query-tile schedule). Return codes as jattn_fwd, plus
 * JATTN_ERR_INVALID for another activation, D != 128 or norm_by_lkv. */
int jattn_fwd_mxfp8(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint8_t* q,
                    const uint8_t* q_scales, const int32_t* q_block_start, const uint8_t* k, const uint8_t* k_scales,
                    const uint8_t* v, const uint8_t* v_scales, const int32_t* kv_block_start, uint16_t* o, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream);

/* MXFP8 attention backward (the same section: block-scaled FP8 MMAs in the
 * backward too, dS quantized online with [32, 32] square blocks so that one
 * quantization serves dS and its transpose).
 *
 * Gradients of jattn_fwd_mxfp8's attention: q, k, v (and their scales and
 * block starts) as there; dout = dO as jattn_mxfp8_quantize output with the
 * query side's offsets (codes [total_q, H, 128] 16-byte aligned, scales
 * [row blocks, H, 4] 4-byte aligned, sharing q_block_start); o (bf16
 * [total_q, H, 128]) and lse (fp32 [total_q, H]) from the forward. Every
 * product is a block-scaled tensor-core MMA on the exact values of its FP8
 * operands with fp32 accumulation:
 *   D_i = <dO~_i, o_i>,  P = exp(s - lse),  dS = P (dP - D),  dP = dO~ V~^T,
 *   dV = P~^T dO~,  dQ = scale dS~ K~,  dK = scale dS~^T Q~,
 * with P~ = P quantized per key and 32-query block with the scale
 * 2^(ceil(log2 x) - 8), x the block's largest P (as the forward), and dS~
 * = dS quantized per [32, 32] block of (query, key) pairs counted from the
 * sequence starts, with the Microscaling rule of jattn_mxfp8_quantize (scale
 * 2^(floor(log2 amax) - 8), saturating at +-448). dq, dk, dv are bf16
 * [total, H, 128], 16-byte aligned; rows that see nothing get zeros. Against
 * the definition with P quantized at the final row maximum (scale 2^-8 of
 * exp(s - m), divided by l), |dv - dv_ref| <= sum_i (2^-3 p_ij + 2^-16 / l_i)
 * |dO~_i| plus bf16 rounding; dq and dk differ from the definition by the
 * quantization steps of dS~ that either side's fp32 rounding can move.
 * The workspace is jattn_bwd's (jattn_workspace_size with act softmax): it
 * holds D and the two tile schedules. The passes run in order D, dQ, dK/dV
 * on `stream`. Return codes as jattn_bwd, plus JATTN_ERR_INVALID for another
 * activation, D != 128 or norm_by_lkv. */
int jattn_bwd_mxfp8(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint8_t* q,
                    const uint8_t* q_scales, const int32_t* q_block_start, const uint8_t* k, const uint8_t* k_scales,
                    const uint8_t* v, const uint8_t* v_scales, const int32_t* kv_block_start, const uint16_t* o,
                    const float* lse, const uint8_t* dout, const uint8_t* dout_scales, uint16_t* dq, uint16_t* dk,
                    uint16_t* dv, void* workspace, size_t workspace_bytes, void* stream);

/* Longest-first tile schedule ("GEM Training" post, GDPA section: valid tiles
 * are precomputed, empty ones skipped, and the rest spread over the SMs so
 * no SM gets a much longer share). Builds the schedule the kernels use into
 * the workspace and copies it to `tiles` (device int32 [max_tiles][4]: b,
 * row tile, first column tile, end column tile) and its length to
 * `n_tiles` (device int32). Rows are query tiles of `row_tile` rows and
 * columns key tiles of `col_tile` rows; with `transposed` the roles swap.
 * Order: column-tile count (capped at 1023) descending, then (b, row tile).
 * max_tiles must be at least jattn_max_tiles(p, row_tile, transposed). */
int jattn_schedule(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, int row_tile,
                   int col_tile, int transposed, int32_t* tiles, int64_t max_tiles, int32_t* n_tiles,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Split of one jagged batch over n_ranks data-parallel ranks (host code;
 * every pointer is a HOST pointer). Sequences are independent problems, so
 * a batch shards by sequence with no exchange inside attention; the cost of
 * a sequence is its number of allowed (query, key) pairs under `mask` /
 * `window` (the jattn_params_t rules), and the split balances that cost the
 * way the GEM training summary's "Base Batch Shuffling" takeaway balances
 * sequence lengths (sort, then spread the heaviest first): sequences in
 * order of decreasing cost (ties: lower index first) each go to the rank
 * with the least cost so far (ties: lower rank). This longest-first greedy
 * rule keeps every rank within one sequence's cost of the mean.
 * q_off, kv_off: int64 [B+1] host prefix sums (off[0] = 0, non-decreasing).
 * rank_of: int32 [B] out, the rank of each sequence. rank_pairs: int64
 * [n_ranks] out, each rank's total allowed pairs per head. Returns
 * JATTN_ERR_INVALID for B outside [1, 2^31), n_ranks < 1, a NULL pointer,
 * an invalid mask or width, or offsets that are not prefix sums. */
int jattn_partition(int64_t B, const int64_t* q_off, const int64_t* kv_off, int mask, int window, int n_ranks,
                    int32_t* rank_of, int64_t* rank_pairs);

/* Upper bound on the number of tiles jattn_schedule can produce. */
int64_t jattn_max_tiles(const jattn_params_t* p, int row_tile, int transposed);

/* Synchronises `stream`, then reads and clears the device status word of
 * `workspace` into *device_status (JATTN_OK or JATTN_ERR_OFFSETS /
 * JATTN_ERR_TIMEOUT). Returns JATTN_ERR_CUDA if the stream reports an error. */
int jattn_get_status(void* workspace, void* stream, int* device_status);

/* Static, human-readable name of a return / status code. */
const char* jattn_error_string(int code);

/* For the calling thread: which CUDA step failed most recently and the
 * runtime's message (empty if none). Valid until the next failing call. */
const char* jattn_last_error(void);

/* Allocation-free forward. No counterpart in the paper: this is a library
 * service. Some callers cannot allocate device memory at the point where
 * they run attention: an application whose memory is carved up in advance by
 * its own pool and that forbids allocations outside it, a plugin invoked by a
 * host runtime that owns all device memory, or a latency-critical serving
 * loop that must never block in the allocator. For them this entry point
 * computes exactly what jattn_fwd computes (same kernels, same results) but
 * takes no workspace: its scratch (the status word and the tile schedule) is
 * a fixed array of JATTN_NOALLOC_SCRATCH_BYTES inside the library, which
 * every GPU that loads the library holds until the process exits. The
 * caller still owns q, k, v, offsets, o and lse (same layout and rules as
 * jattn_fwd) and may pass `device_status`, a device int that receives the
 * status word (JATTN_OK / JATTN_ERR_OFFSETS / JATTN_ERR_TIMEOUT) once the
 * call's work on `stream` completes; NULL skips it.
 *
 * Limits and rules:
 *  - The schedule needs about 48 bytes per 256 query rows plus 4 bytes per
 *    sequence: 256 + 4*(B+1) + 48*(total_q/256 + B + 1) bytes, rounded up
 *    per buffer. Calls that need more return JATTN_ERR_TOO_LARGE (and
 *    jattn_last_error says how much) without launching anything.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture. The array has its own address in every CUDA
 *    context, so the address is cached together with the id of the context
 *    current at the call (cuCtxGetId), and a call made under another context
 *    of the device (a runtime that owns its contexts, or the primary context
 *    created again after cudaDeviceReset) looks it up again: make the first
 *    call under each context before any capture on it too.
 *  - Every call reuses the same array; each call clears the status word
 *    first. Calls whose work overlaps on the GPU (other streams, other host
 *    threads) race on the array: serialise them.
 *  - No cudaMalloc, cudaFree or other allocating call is made. */
#define JATTN_NOALLOC_SCRATCH_BYTES (8u << 20)
int jattn_fwd_noalloc(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint16_t* q,
                      const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse, int* device_status,
                      void* stream);

/* Profiling hook, per host thread: `events` points to six cudaEvent_t
 * (passed as void*) that later calls made from the calling thread record on
 * their stream (calls from other threads record nothing): events[0] / [1]
 * right before / after the forward kernel launch, [2] / [3] around the dK/dV
 * kernel, [4] / [5] around the dQ kernel (which jattn_bwd launches first);
 * NULL turns it off. The library keeps the handles, not copies: turn the hook
 * off before destroying the events. Used to time those kernels with events
 * on the stream they run on. */
void jattn_profile_events(void* const* events);

/* Test hook, per host thread (launches made from other threads keep their
 * own settings): after this call, bounded waits in the kernels give up after
 * `timeout_ns` nanoseconds (0 restores the default of two seconds), and
 * flag bit 0 makes the next launches skip the query-tile copy so that the
 * first wait on it runs out. Used to check that an expired wait reports
 * JATTN_ERR_TIMEOUT and leaves the context usable. Flag bit 1 (bit 2) makes
 * the forward use the column-split (ping-pong) arrangement of its activation
 * warps whatever the shapes, so both can be checked on the same inputs;
 * results agree within floating-point rounding order. The other bits pick
 * between code paths that compute the same results in the same way: bit 3
 * (bit 4) makes the dQ pass hold K and V in two rings (one ring); bit 5 runs
 * pooling and short-key shapes on the general kernels; bit 6 runs the
 * short-key shapes' forward on the short-query (keys-on-M) kernel; bit 7 runs
 * their backward on the short-query backward's cross mode (64-query chunks). */
void jattn_debug_set(int flags, uint64_t timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* JATTN_H */
