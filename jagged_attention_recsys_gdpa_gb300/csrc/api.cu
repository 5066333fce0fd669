// C-ABI entry points of libjattn: argument checks, workspace layout, TMA
// descriptors and kernel launches on the caller's stream.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/jattn.h"
#include "common.cuh"
#include "kernels.h"
#include "sched.h"

namespace jattn {
namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
thread_local char g_last_error[256] = "";
// Test and profiling hooks are per host thread: a hook set on one thread
// never changes the launches another thread makes.
thread_local int g_debug_flags = 0;

// Key tiles a 128-row query tile visits on average, from the mask and the
// mean key length: with a window, min(W, L) / 128 + 1; causal, L / 256 + 1;
// none, L / 128 + 1; a block mask (blocks dividing the tile), one.
double key_tiles_per_query_tile(const jattn_params_t& p) {
  if (p.B < 1) return 0.0;
  if (p.mask & JATTN_MASK_BLOCK) return 1.0;
  const double lkv = static_cast<double>(p.total_kv) / static_cast<double>(p.B);
  if (p.mask & JATTN_MASK_WINDOW) return std::min(static_cast<double>(p.window), lkv) / 128.0 + 1.0;
  if (p.mask & JATTN_MASK_CAUSAL) return lkv / 256.0 + 1.0;
  return lkv / 128.0 + 1.0;
}

// Forward activation arrangement: the column split when sequences average at
// most one 128-row query tile (most items then hold a single tile) or query
// tiles visit fewer than six key tiles (windows, blocks: the split's two
// warpgroups finish each tile's softmax sooner, which matters more than the
// ping-pong's overlap over so few tiles), else the ping-pong between two
// query tiles. Debug flag bits 1 / 2 force either one.
bool fwd_split(const jattn_params_t& p) {
  if (g_debug_flags & 2) return true;
  if (g_debug_flags & 4) return false;
  return p.total_q <= static_cast<int64_t>(kTile) * p.B || key_tiles_per_query_tile(p) < 6.0;
}
thread_local uint64_t g_timeout_ns = kDefaultTimeoutNs;
// Optional events recorded around the main kernels: [fwd, dkdv, dq] x [begin, end].
thread_local cudaEvent_t g_prof[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};

void prof(int i, cudaStream_t st) {
  if (g_prof[i]) cudaEventRecord(g_prof[i], st);
}

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Record which CUDA step failed (readable through jattn_last_error).
int cuda_fail(const char* what, cudaError_t e) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
  return JATTN_ERR_CUDA;
}

// Errors left by earlier, unrelated runtime calls on this thread must not be
// mistaken for a failed launch of ours.
void clear_stale_error() { (void)cudaGetLastError(); }

// Pointwise attention without a mask at D = 128 runs on the kernels of
// pma.cu when its sequences are short on one side: pooling (at most 64
// queries per sequence on average: the keys-on-M forward and the fused
// backward) or cross-attention over short key sequences (at most 128 keys per
// sequence on average: the short-key forward and the fused backward). The
// workspace holds their schedule and gate word whenever the shape allows
// them. Debug flag bit 32 keeps the general kernels; bit 64 runs the
// short-key shapes' forward on the short-query kernel (for comparisons).
bool pointwise_unmasked(const jattn_params_t& p) {
  return p.act != JATTN_SOFTMAX && p.mask == JATTN_MASK_NONE && p.D == 128;
}
bool short_q_shape(const jattn_params_t& p) {
  return pointwise_unmasked(p) && p.total_q <= static_cast<int64_t>(pma_rows_per_item()) * p.B;
}
bool short_kv_shape(const jattn_params_t& p) {
  return pointwise_unmasked(p) && !short_q_shape(p) && p.total_kv <= static_cast<int64_t>(kTile) * p.B;
}
bool use_short_q(const jattn_params_t& p) { return short_q_shape(p) && !(g_debug_flags & 32); }
bool use_short_kv(const jattn_params_t& p) { return short_kv_shape(p) && !(g_debug_flags & 32); }
bool use_short_q_fwd(const jattn_params_t& p) {
  return use_short_q(p) || (use_short_kv(p) && (g_debug_flags & 64));
}

struct Layout {
  size_t status, sched_fwd, sched_q, sched_kv, sched_s, gate, di, lse, total;
  int64_t tiles_fwd, tiles_q, tiles_kv, tiles_s;
};

Layout layout_for(const jattn_params_t& p) {
  Layout L{};
  const int fwd_rows = fwd_rows_per_item();
  L.tiles_fwd = sched_max_tiles(p.B, p.total_q, fwd_rows);
  L.tiles_q = sched_max_tiles(p.B, p.total_q, kTile);
  L.tiles_kv = sched_max_tiles(p.B, p.total_kv, kTile);
  size_t off = 0;
  L.status = off;
  off += 256;
  L.sched_fwd = off;
  off += al256(sched_ws_bytes(p.B, L.tiles_fwd));
  L.sched_q = off;
  off += al256(sched_ws_bytes(p.B, L.tiles_q));
  L.sched_kv = off;
  off += al256(sched_ws_bytes(p.B, L.tiles_kv));
  L.sched_s = L.gate = off;
  L.tiles_s = 0;
  if (short_q_shape(p) || short_kv_shape(p)) {
    // pooling: 64-row query tiles; cross: 128-row key tiles (and, under debug
    // flag bit 64, the forward's 64-row query tiles)
    L.tiles_s = std::max(sched_max_tiles(p.B, p.total_q, pma_rows_per_item()),
                         short_kv_shape(p) ? sched_max_tiles(p.B, p.total_kv, kTile) : int64_t(0));
    off += al256(sched_ws_bytes(p.B, L.tiles_s));
    L.gate = off;
    off += 256;
  }
  L.di = off;
  if (p.act == JATTN_SOFTMAX) off += al256(sizeof(float) * static_cast<size_t>(p.total_q) * p.H);
  // block masks: the LSE that a backward with in-tile statistics writes for its dK/dV pass
  L.lse = off;
  if (p.act == JATTN_SOFTMAX && (p.mask & JATTN_MASK_BLOCK))
    off += al256(sizeof(float) * static_cast<size_t>(p.total_q) * p.H);
  L.total = off;
  return L;
}

// BlockAttention with blocks that divide the 128-row tile, on self-attention
// (one offsets array for both sides, so every sequence has delta = 0): every
// query tile then meets exactly one key tile, so the backward takes the
// softmax statistics and Di from that tile and needs neither O nor LSE.
bool block_in_tile(const jattn_params_t& p, const int64_t* q_off, const int64_t* kv_off) {
  return p.act == JATTN_SOFTMAX && (p.mask & JATTN_MASK_BLOCK) && p.window >= 1 && kTile % p.window == 0 &&
         q_off == kv_off && p.total_q == p.total_kv;
}

int check_params(const jattn_params_t* p) {
  if (!p) return JATTN_ERR_INVALID;
  if (p->B < 1 || p->total_q < 0 || p->total_kv < 0 || p->H < 1) return JATTN_ERR_INVALID;
  // The schedule keeps sequence indices and per-sequence tile counts in 32 bits.
  if (p->B >= (int64_t(1) << 31)) return JATTN_ERR_INVALID;
  if (p->D != 64 && p->D != 128) return JATTN_ERR_INVALID;
  if (p->act != JATTN_SOFTMAX && p->act != JATTN_SILU && p->act != JATTN_GELU_TANH && p->act != JATTN_GELU_POLY)
    return JATTN_ERR_INVALID;
  if (p->mask != JATTN_MASK_NONE && p->mask != JATTN_MASK_CAUSAL &&
      p->mask != (JATTN_MASK_CAUSAL | JATTN_MASK_WINDOW) && p->mask != JATTN_MASK_BLOCK &&
      p->mask != (JATTN_MASK_CAUSAL | JATTN_MASK_BLOCK))
    return JATTN_ERR_INVALID;
  if ((p->mask & (JATTN_MASK_WINDOW | JATTN_MASK_BLOCK)) && p->window < 1) return JATTN_ERR_INVALID;
  if (!(p->scale >= 0.0f) || !std::isfinite(p->scale)) return JATTN_ERR_INVALID;
  if (p->norm_by_lkv != 0 && p->norm_by_lkv != 1) return JATTN_ERR_INVALID;
  if (p->norm_by_lkv && p->act == JATTN_SOFTMAX) return JATTN_ERR_INVALID;
  // TMA row coordinates and per-sequence row indices are 32-bit.
  if (p->total_q >= (int64_t(1) << 31) || p->total_kv >= (int64_t(1) << 31)) return JATTN_ERR_INVALID;
  if (static_cast<int64_t>(p->H) * p->D * 2 >= (int64_t(1) << 31)) return JATTN_ERR_INVALID;
  return JATTN_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }
bool aligned32(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 31u) == 0; }

int check_ws(const jattn_params_t* p, void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return JATTN_ERR_WORKSPACE;
  if (ws_bytes < layout_for(*p).total) return JATTN_ERR_WORKSPACE;
  return JATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};
DeviceInfo g_dev[64];
std::mutex g_dev_mu;

int device_info(DeviceInfo& out) {
  int dev = 0;
  cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 != cudaSuccess) return cuda_fail("cudaGetDevice", e0);
  if (dev < 0 || dev >= 64) return JATTN_ERR_CUDA;
  // Make the device's primary context current on this thread (a fresh thread,
  // e.g. an autograd worker, may have none yet; tensor-map encoding needs it).
  if ((e0 = cudaSetDevice(dev)) != cudaSuccess) return cuda_fail("cudaSetDevice", e0);
  std::lock_guard<std::mutex> g(g_dev_mu);
  if (!g_dev[dev].ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cuda_fail("cudaDeviceGetAttribute", cudaGetLastError());
    if (major != 10 || minor != 3) return JATTN_ERR_UNSUPPORTED;
    g_dev[dev].sms = sms;
    g_dev[dev].ok = true;
  }
  out = g_dev[dev];
  return JATTN_OK;
}

int encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? JATTN_OK : JATTN_ERR_CUDA;
}

// 2-D view [rows, H*D] of a jagged bf16 tensor; boxes of box_rows rows x 64
// columns (128 bytes) with the 128-byte swizzle the MMA descriptors expect.
int make_map(CUtensorMap* m, const void* ptr, int64_t rows, int H, int D, int box_rows = kTile) {
  std::memset(m, 0, sizeof(*m));
  if (rows == 0) return JATTN_OK;  // never dereferenced: no tile is scheduled
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * D, static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * D * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? JATTN_OK : JATTN_ERR_CUDA;
}

// Pointwise activations without the 1/Lkv normaliser: P and dS enter the
// second products as two bf16 parts (hi = bf16(x), lo = bf16(x - hi)) that
// accumulate into the same fp32 result, so their rounding does not grow with
// the sequence length (outputs there sum thousands of unscaled terms).
bool hilo_for(const jattn_params_t& p) { return p.act != JATTN_SOFTMAX && !p.norm_by_lkv; }

// The dQ pass's K / V layout: two rings (K deeper than V) when query tiles
// see many key tiles on average (six or more), where each tile's K latency
// would otherwise show, one ring otherwise, where the second ring's barrier
// and release cost more than they hide. Debug flag bits 8 / 16 force two
// rings / one ring.
bool dq_split_rings(const jattn_params_t& p) {
  if (g_debug_flags & 8) return true;
  if (g_debug_flags & 16) return false;
  if (p.B < 1 || (p.mask & JATTN_MASK_BLOCK)) return false;
  return key_tiles_per_query_tile(p) >= 6.0;
}

// 2-D view [rows, H*D] of jagged E4M3 codes (one byte each); boxes of
// box_rows rows x 128 bytes with the 128-byte swizzle (D = 128: one box per
// head row).
int make_map_u8(CUtensorMap* m, const void* ptr, int64_t rows, int H, int D, int box_rows = kTile) {
  std::memset(m, 0, sizeof(*m));
  if (rows == 0) return JATTN_OK;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * D, static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * D};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? JATTN_OK : JATTN_ERR_CUDA;
}

AttnArgs base_args(const jattn_params_t& p, const int64_t* q_off, const int64_t* kv_off, void* ws) {
  AttnArgs a{};
  a.q_off = q_off;
  a.kv_off = kv_off;
  a.H = p.H;
  a.mask = p.mask;
  a.window = (p.mask & (JATTN_MASK_WINDOW | JATTN_MASK_BLOCK)) ? p.window : 0;
  const float scale = p.scale > 0.0f ? p.scale : 1.0f / std::sqrt(static_cast<float>(p.D));
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.norm_by_lkv = p.norm_by_lkv;
  a.status = reinterpret_cast<DevStatus*>(static_cast<char*>(ws));
  a.timeout_ns = g_timeout_ns;
  a.debug_flags = g_debug_flags;
  return a;
}

int grid_for(const DeviceInfo& d, int64_t max_tiles, int H) {
  const int64_t items = max_tiles * H;
  return static_cast<int>(items < d.sms ? (items > 0 ? items : 1) : d.sms);
}

}  // namespace
}  // namespace jattn

// ---------------------------------------------------------------- allocation-free forward
// Scratch of jattn_fwd_noalloc (status word + forward tile schedule), held in
// the library's own device memory so that its callers allocate nothing.
static __device__ __align__(256) unsigned char jattn_noalloc_scratch[JATTN_NOALLOC_SCRATCH_BYTES];

namespace jattn {
namespace {

// Device address of the scratch array. A module-scope __device__ array has
// its own address in every CUDA context (and a new one after a context is
// destroyed and created again), so the address is looked up with the device
// current and cached per device together with the id of the context it
// belongs to (cuCtxGetId: unique for the life of the process); a call from
// another context of the same device looks it up again. Host code may not
// use the symbol itself as an address.
struct NoallocSlot {
  unsigned long long ctx_id;
  void* addr;
};
NoallocSlot g_noalloc[64] = {};
std::mutex g_noalloc_mu;

typedef CUresult (*PFN_ctx_get_current)(CUcontext*);
typedef CUresult (*PFN_ctx_get_id)(CUcontext, unsigned long long*);
PFN_ctx_get_current g_ctx_current = nullptr;
PFN_ctx_get_id g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Id of the context current on this thread (device_info has made the
// device's primary context current if there was none).
int current_ctx_id(unsigned long long* id) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_ctx_get_current>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_ctx_get_id>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) {
    snprintf(g_last_error, sizeof(g_last_error), "driver entry points cuCtxGetCurrent / cuCtxGetId not found");
    return JATTN_ERR_CUDA;
  }
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || g_ctx_id(ctx, id) != CUDA_SUCCESS) {
    snprintf(g_last_error, sizeof(g_last_error), "no current CUDA context for the scratch lookup");
    return JATTN_ERR_CUDA;
  }
  return JATTN_OK;
}

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= 64) return JATTN_ERR_CUDA;
  unsigned long long id = 0;
  const int rc = current_ctx_id(&id);
  if (rc != JATTN_OK) return rc;
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (!g_noalloc[dev].addr || g_noalloc[dev].ctx_id != id) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, jattn_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress", e);
    g_noalloc[dev].addr = ptr;
    g_noalloc[dev].ctx_id = id;
  }
  *out = g_noalloc[dev].addr;
  return JATTN_OK;
}

}  // namespace
}  // namespace jattn

using namespace jattn;

extern "C" {

int jattn_workspace_size(const jattn_params_t* p, size_t* bytes) {
  if (!bytes) return JATTN_ERR_INVALID;
  const int rc = check_params(p);
  if (rc != JATTN_OK) return rc;
  *bytes = layout_for(*p).total;
  return JATTN_OK;
}

int64_t jattn_max_tiles(const jattn_params_t* p, int row_tile, int transposed) {
  if (check_params(p) != JATTN_OK || row_tile < 1) return -1;
  return sched_max_tiles(p->B, transposed ? p->total_kv : p->total_q, row_tile);
}

int jattn_fwd(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint16_t* q,
              const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse, void* ws, size_t ws_bytes,
              void* stream) {
  int rc = check_params(p);
  if (rc != JATTN_OK) return rc;
  if (!q_off || !kv_off) return JATTN_ERR_INVALID;
  if ((p->total_q > 0 && (!q || !o)) || (p->total_kv > 0 && (!k || !v))) return JATTN_ERR_INVALID;
  if (p->act == JATTN_SOFTMAX && p->total_q > 0 && !lse && !(p->mask & JATTN_MASK_BLOCK)) return JATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return JATTN_ERR_ALIGN;
  if ((rc = check_ws(p, ws, ws_bytes)) != JATTN_OK) return rc;
  DeviceInfo dev;
  if ((rc = device_info(dev)) != JATTN_OK) return rc;
  if ((rc = encoder()) != JATTN_OK) return rc;
  clear_stale_error();
  if (p->total_q == 0) return JATTN_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = layout_for(*p);
  char* base = static_cast<char*>(ws);
  AttnArgs a = base_args(*p, q_off, kv_off, ws);
  cudaError_t e;
  if (use_short_q_fwd(*p)) {
    const SchedView ss = sched_carve(base + L.sched_s, p->B, L.tiles_s);
    if ((e = sched_launch(ss, q_off, kv_off, p->B, p->total_q, p->total_kv, pma_rows_per_item(), kTile, p->mask,
                          a.window, 0, a.status, st)) != cudaSuccess)
      return cuda_fail("schedule launch", e);
    CUtensorMap mq, mk, mv;
    if (make_map(&mq, q, p->total_q, p->H, p->D, pma_rows_per_item()) ||
        make_map(&mk, k, p->total_kv, p->H, p->D) || make_map(&mv, v, p->total_kv, p->H, p->D))
      return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
    a.tiles = ss.sorted;
    a.n_tiles = ss.n_tiles;
    a.out0 = reinterpret_cast<__nv_bfloat16*>(o);
    a.out_v8 = aligned32(o);
    prof(0, st);
    if ((e = launch_pma_fwd(p->act, hilo_for(*p), mq, mk, mv, a, grid_for(dev, L.tiles_s, p->H), st)) !=
        cudaSuccess)
      return cuda_fail("short-query forward kernel launch", e);
    prof(1, st);
    return JATTN_OK;
  }
  const SchedView sv = sched_carve(base + L.sched_fwd, p->B, L.tiles_fwd);
  if ((e = sched_launch(sv, q_off, kv_off, p->B, p->total_q, p->total_kv, fwd_rows_per_item(), kTile, p->mask,
                        a.window, 0, a.status, st)) != cudaSuccess)
    return cuda_fail("schedule launch", e);
  CUtensorMap mq, mk, mv;
  if (make_map(&mq, q, p->total_q, p->H, p->D) || make_map(&mk, k, p->total_kv, p->H, p->D) ||
      make_map(&mv, v, p->total_kv, p->H, p->D))
    return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
  a.out0 = reinterpret_cast<__nv_bfloat16*>(o);
  a.f0 = lse;
  a.out_v8 = aligned32(o);
  prof(0, st);
  // Cross-attention over short key sequences: the short-key forward runs first
  // and, when the gate finds every sequence within 128 keys, the general
  // forward below finds an empty schedule.
  if (use_short_kv(*p) && p->total_kv > 0) {
    const SchedView ss = sched_carve(base + L.sched_s, p->B, L.tiles_s);
    if ((e = sched_launch(ss, q_off, kv_off, p->B, p->total_q, p->total_kv, kTile, kTile, p->mask, a.window, 1,
                          a.status, st)) != cudaSuccess)
      return cuda_fail("schedule launch", e);
    int* gate = reinterpret_cast<int*>(base + L.gate);
    if ((e = launch_pma_gate(q_off, kv_off, p->B, true, gate, sv.n_tiles, sv.n_tiles, st)) != cudaSuccess)
      return cuda_fail("short-key gate launch", e);
    AttnArgs b = a;
    b.tiles = ss.sorted;
    b.n_tiles = ss.n_tiles;
    if ((e = launch_skv_fwd(p->act, hilo_for(*p), mq, mk, mv, b, gate, grid_for(dev, L.tiles_s, p->H), st)) !=
        cudaSuccess)
      return cuda_fail("short-key forward kernel launch", e);
  }
  a.tiles = sv.sorted;
  a.n_tiles = sv.n_tiles;
  if ((e = launch_fwd(p->D, p->act, fwd_split(*p), (p->mask & JATTN_MASK_BLOCK) != 0, hilo_for(*p), mq, mk, mv, a,
                        grid_for(dev, L.tiles_fwd, p->H), st)) != cudaSuccess)
    return cuda_fail("forward kernel launch", e);
  prof(1, st);
  return JATTN_OK;
}

int jattn_fwd_noalloc(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint16_t* q,
                      const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse, int* device_status,
                      void* stream) {
  int rc = check_params(p);
  if (rc != JATTN_OK) return rc;
  if (!q_off || !kv_off) return JATTN_ERR_INVALID;
  if ((p->total_q > 0 && (!q || !o)) || (p->total_kv > 0 && (!k || !v))) return JATTN_ERR_INVALID;
  if (p->act == JATTN_SOFTMAX && p->total_q > 0 && !lse) return JATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return JATTN_ERR_ALIGN;
  const Layout L = layout_for(*p);
  const size_t need = 256 + sched_ws_bytes(p->B, L.tiles_fwd);
  if (need > JATTN_NOALLOC_SCRATCH_BYTES) {
    snprintf(g_last_error, sizeof(g_last_error), "jattn_fwd_noalloc needs %zu bytes of scratch; the library holds %zu",
             need, static_cast<size_t>(JATTN_NOALLOC_SCRATCH_BYTES));
    return JATTN_ERR_TOO_LARGE;
  }
  DeviceInfo dev;
  if ((rc = device_info(dev)) != JATTN_OK) return rc;
  if ((rc = encoder()) != JATTN_OK) return rc;
  void* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch)) != JATTN_OK) return rc;
  clear_stale_error();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  // The status word must start at zero; the schedule buffers are fully rewritten.
  if ((e = cudaMemsetAsync(scratch, 0, 256, st)) != cudaSuccess) return cuda_fail("status clear", e);
  if (p->total_q > 0) {
    char* base = static_cast<char*>(scratch);
    const SchedView sv = sched_carve(base + 256, p->B, L.tiles_fwd);
    AttnArgs a = base_args(*p, q_off, kv_off, scratch);
    if ((e = sched_launch(sv, q_off, kv_off, p->B, p->total_q, p->total_kv, fwd_rows_per_item(), kTile, p->mask,
                          a.window, 0, a.status, st)) != cudaSuccess)
      return cuda_fail("schedule launch", e);
    CUtensorMap mq, mk, mv;
    if (make_map(&mq, q, p->total_q, p->H, p->D) || make_map(&mk, k, p->total_kv, p->H, p->D) ||
        make_map(&mv, v, p->total_kv, p->H, p->D))
      return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
    a.tiles = sv.sorted;
    a.n_tiles = sv.n_tiles;
    a.out0 = reinterpret_cast<__nv_bfloat16*>(o);
    a.f0 = lse;
    a.out_v8 = aligned32(o);
    if ((e = launch_fwd(p->D, p->act, fwd_split(*p), (p->mask & JATTN_MASK_BLOCK) != 0, hilo_for(*p), mq, mk, mv, a,
                        grid_for(dev, L.tiles_fwd, p->H), st)) != cudaSuccess)
      return cuda_fail("forward kernel launch", e);
  }
  if (device_status &&
      (e = cudaMemcpyAsync(device_status, scratch, sizeof(int), cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
    return cuda_fail("status copy", e);
  return JATTN_OK;
}

int jattn_fwd_mxfp8(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint8_t* q,
                    const uint8_t* q_scales, const int32_t* q_block_start, const uint8_t* k, const uint8_t* k_scales,
                    const uint8_t* v, const uint8_t* v_scales, const int32_t* kv_block_start, uint16_t* o, float* lse,
                    void* ws, size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc != JATTN_OK) return rc;
  if (p->act != JATTN_SOFTMAX || p->D != 128 || p->norm_by_lkv) return JATTN_ERR_INVALID;
  if (!q_off || !kv_off || !q_block_start || !kv_block_start) return JATTN_ERR_INVALID;
  if (p->total_q > 0 && (!q || !q_scales || !o || !lse)) return JATTN_ERR_INVALID;
  if (p->total_kv > 0 && (!k || !k_scales || !v || !v_scales)) return JATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return JATTN_ERR_ALIGN;
  auto aligned4 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 3u) == 0; };
  if (!aligned4(q_scales) || !aligned4(k_scales) || !aligned4(v_scales)) return JATTN_ERR_ALIGN;
  if ((rc = check_ws(p, ws, ws_bytes)) != JATTN_OK) return rc;
  DeviceInfo dev;
  if ((rc = device_info(dev)) != JATTN_OK) return rc;
  if ((rc = encoder()) != JATTN_OK) return rc;
  clear_stale_error();
  if (p->total_q == 0) return JATTN_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = layout_for(*p);
  const SchedView sv = sched_carve(static_cast<char*>(ws) + L.sched_q, p->B, L.tiles_q);
  AttnArgs a = base_args(*p, q_off, kv_off, ws);
  cudaError_t e;
  if ((e = sched_launch(sv, q_off, kv_off, p->B, p->total_q, p->total_kv, kTile, kTile, p->mask, a.window, 0,
                        a.status, st)) != cudaSuccess)
    return cuda_fail("schedule launch", e);
  CUtensorMap mq, mk, mv;
  if (make_map_u8(&mq, q, p->total_q, p->H, p->D) || make_map_u8(&mk, k, p->total_kv, p->H, p->D) ||
      make_map_u8(&mv, v, p->total_kv, p->H, p->D))
    return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
  a.tiles = sv.sorted;
  a.n_tiles = sv.n_tiles;
  a.out0 = reinterpret_cast<__nv_bfloat16*>(o);
  a.f0 = lse;
  a.out_v8 = aligned32(o);
  a.sf_q = q_scales;
  a.sf_k = k_scales;
  a.sf_v = v_scales;
  a.bs_q = q_block_start;
  a.bs_kv = kv_block_start;
  prof(0, st);
  if ((e = launch_fwd_mx(mq, mk, mv, a, grid_for(dev, L.tiles_q, p->H), st)) != cudaSuccess)
    return cuda_fail("MXFP8 forward kernel launch", e);
  prof(1, st);
  return JATTN_OK;
}

int jattn_bwd_mxfp8(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint8_t* q,
                    const uint8_t* q_scales, const int32_t* q_block_start, const uint8_t* k, const uint8_t* k_scales,
                    const uint8_t* v, const uint8_t* v_scales, const int32_t* kv_block_start, const uint16_t* o,
                    const float* lse, const uint8_t* dout, const uint8_t* dout_scales, uint16_t* dq, uint16_t* dk,
                    uint16_t* dv, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc != JATTN_OK) return rc;
  if (p->act != JATTN_SOFTMAX || p->D != 128 || p->norm_by_lkv) return JATTN_ERR_INVALID;
  if (!q_off || !kv_off || !q_block_start || !kv_block_start) return JATTN_ERR_INVALID;
  if (p->total_q > 0 && (!q || !q_scales || !o || !lse || !dout || !dout_scales || !dq)) return JATTN_ERR_INVALID;
  if (p->total_kv > 0 && (!k || !k_scales || !v || !v_scales || !dk || !dv)) return JATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return JATTN_ERR_ALIGN;
  auto aligned4 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 3u) == 0; };
  if (!aligned4(q_scales) || !aligned4(k_scales) || !aligned4(v_scales) || !aligned4(dout_scales))
    return JATTN_ERR_ALIGN;
  if ((rc = check_ws(p, ws, ws_bytes)) != JATTN_OK) return rc;
  DeviceInfo dev;
  if ((rc = device_info(dev)) != JATTN_OK) return rc;
  if ((rc = encoder()) != JATTN_OK) return rc;
  clear_stale_error();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  const Layout L = layout_for(*p);
  AttnArgs a = base_args(*p, q_off, kv_off, ws);
  float* di = reinterpret_cast<float*>(base + L.di);
  cudaError_t e;
  CUtensorMap mq, mk, mv, mdo, mq96, mdo96;
  if (make_map_u8(&mq, q, p->total_q, p->H, p->D) || make_map_u8(&mk, k, p->total_kv, p->H, p->D) ||
      make_map_u8(&mv, v, p->total_kv, p->H, p->D) || make_map_u8(&mdo, dout, p->total_q, p->H, p->D) ||
      make_map_u8(&mq96, q, p->total_q, p->H, p->D, 96) || make_map_u8(&mdo96, dout, p->total_q, p->H, p->D, 96))
    return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
  a.f0 = const_cast<float*>(lse);
  a.f1 = di;
  a.sf_q = q_scales;
  a.sf_k = k_scales;
  a.sf_v = v_scales;
  a.sf_do = dout_scales;
  a.bs_q = q_block_start;
  a.bs_kv = kv_block_start;
  // D first: both passes read it
  if (p->total_q > 0) {
    if ((e = launch_mx_di(q_off, static_cast<int>(p->B), p->H, jattn_mxfp8_scale_rows(p->B, p->total_q), dout,
                          dout_scales, q_block_start, o, di, st)) != cudaSuccess)
      return cuda_fail("D kernel launch", e);
    const SchedView qs = sched_carve(base + L.sched_q, p->B, L.tiles_q);
    if ((e = sched_launch(qs, q_off, kv_off, p->B, p->total_q, p->total_kv, kTile, kTile, p->mask, a.window, 0,
                          a.status, st)) != cudaSuccess)
      return cuda_fail("query-tile schedule launch", e);
    a.tiles = qs.sorted;
    a.n_tiles = qs.n_tiles;
    a.out0 = reinterpret_cast<__nv_bfloat16*>(dq);
    a.out1 = nullptr;
    a.out_v8 = aligned32(dq);
    prof(4, st);
    if ((e = launch_bwd_dq_mx(mq, mk, mv, mdo, a, grid_for(dev, L.tiles_q, p->H), st)) != cudaSuccess)
      return cuda_fail("MXFP8 dQ kernel launch", e);
    prof(5, st);
  }
  if (p->total_kv > 0) {
    const SchedView kv = sched_carve(base + L.sched_kv, p->B, L.tiles_kv);
    if ((e = sched_launch(kv, q_off, kv_off, p->B, p->total_q, p->total_kv, kTile, kTile, p->mask, a.window, 1,
                          a.status, st)) != cudaSuccess)
      return cuda_fail("key-tile schedule launch", e);
    a.tiles = kv.sorted;
    a.n_tiles = kv.n_tiles;
    a.out0 = reinterpret_cast<__nv_bfloat16*>(dk);
    a.out1 = reinterpret_cast<__nv_bfloat16*>(dv);
    a.out_v8 = aligned32(dk) && aligned32(dv);
    prof(2, st);
    if ((e = launch_bwd_dkdv_mx(mq96, mk, mv, mdo96, a, grid_for(dev, L.tiles_kv, p->H), st)) != cudaSuccess)
      return cuda_fail("MXFP8 dK/dV kernel launch", e);
    prof(3, st);
  }
  return JATTN_OK;
}

namespace jattn {
namespace {

// Rotary tables: both present, 16-byte aligned, 1 <= rows <= INT_MAX.
int check_rope(const float* c, const float* s, int64_t rows) {
  if (!c || !s || rows < 1 || rows > INT32_MAX) return JATTN_ERR_INVALID;
  if (!aligned16(c) || !aligned16(s)) return JATTN_ERR_ALIGN;
  return JATTN_OK;
}

// Bytes of the pair-major table copies jattn_bwd_rope keeps after the
// workspace's regular layout (256-byte rounded).
size_t rope_extra_bytes(int D, int64_t rows) {
  return (static_cast<size_t>(rows) * D * sizeof(float) + 255) & ~static_cast<size_t>(255);
}

// jattn_bwd and jattn_bwd_rope (rope_cos == nullptr: no rotation).
int bwd_impl(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint16_t* q,
             const uint16_t* k, const uint16_t* v, const uint16_t* o, const float* lse, const uint16_t* dout,
             const float* rope_cos, const float* rope_sin, int64_t rope_rows, uint16_t* dq, uint16_t* dk,
             uint16_t* dv, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc != JATTN_OK) return rc;
  if (!q_off || !kv_off) return JATTN_ERR_INVALID;
  if (p->total_q > 0 && (!q || !dout || !dq)) return JATTN_ERR_INVALID;
  if (p->total_kv > 0 && (!k || !v || !dk || !dv)) return JATTN_ERR_INVALID;
  const bool in_tile = block_in_tile(*p, q_off, kv_off);
  if (p->act == JATTN_SOFTMAX && p->total_q > 0 && !in_tile && (!o || !lse)) return JATTN_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return JATTN_ERR_ALIGN;
  if ((rc = check_ws(p, ws, ws_bytes)) != JATTN_OK) return rc;
  const Layout L = layout_for(*p);
  if (in_tile) o = nullptr;  // neither O nor the forward's LSE is read
  if (rope_cos && ws_bytes < L.total + rope_extra_bytes(p->D, rope_rows)) return JATTN_ERR_WORKSPACE;
  DeviceInfo dev;
  if ((rc = device_info(dev)) != JATTN_OK) return rc;
  if ((rc = encoder()) != JATTN_OK) return rc;
  clear_stale_error();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  AttnArgs a = base_args(*p, q_off, kv_off, ws);
  cudaError_t e;
  if (rope_cos) {
    // pair-major copies of the tables after the regular layout (L.total is 256-byte aligned)
    float* cos_pm = reinterpret_cast<float*>(base + L.total);
    float* sin_pm = cos_pm + static_cast<size_t>(rope_rows) * (p->D / 2);
    if ((e = launch_rope_transpose(rope_cos, rope_sin, static_cast<int>(rope_rows), p->D / 2, cos_pm, sin_pm,
                                   st)) != cudaSuccess)
      return cuda_fail("rotary table transpose launch", e);
    a.rope_cos = cos_pm;
    a.rope_sin = sin_pm;
    a.rope_rows = static_cast<int>(rope_rows);
  }
  float* di = (p->act == JATTN_SOFTMAX) ? reinterpret_cast<float*>(base + L.di) : nullptr;
  CUtensorMap mq, mk, mv, mdo, mo;
  std::memset(&mo, 0, sizeof(mo));  // softmax only: the O tiles the dQ pass reads for Di (one-ring layout)
  if (make_map(&mq, q, p->total_q, p->H, p->D) || make_map(&mk, k, p->total_kv, p->H, p->D) ||
      make_map(&mv, v, p->total_kv, p->H, p->D) || make_map(&mdo, dout, p->total_q, p->H, p->D) ||
      (p->act == JATTN_SOFTMAX && !in_tile && make_map(&mo, o, p->total_q, p->H, p->D)))
    return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
  // softmax: the rows of O the dQ pass reads for Di (two-ring layout)
  a.in0 = (p->act == JATTN_SOFTMAX && !in_tile) ? reinterpret_cast<const __nv_bfloat16*>(o) : nullptr;
  // in-tile statistics: the dQ pass writes LSE and Di into the workspace for the dK/dV pass
  a.f0 = in_tile ? reinterpret_cast<float*>(base + L.lse) : const_cast<float*>(lse);
  a.f1 = di;
  a.in_tile_stats = in_tile ? 1 : 0;
  const SchedView qs = sched_carve(base + L.sched_q, p->B, L.tiles_q);
  const SchedView kv = sched_carve(base + L.sched_kv, p->B, L.tiles_kv);
  // Short-query (pooling) and short-key (cross) shapes: the fused pass runs
  // first and, when the gate finds every sequence within its mode's limits,
  // the general passes below find empty schedules. The profiling events of
  // the dK/dV slot bracket it.
  const bool cross = use_short_kv(*p);
  const bool sq = (use_short_q(*p) || cross) && !rope_cos && p->total_q > 0 && p->total_kv > 0;
  if (sq) {
    const SchedView ss = sched_carve(base + L.sched_s, p->B, L.tiles_s);
    // pooling: 64-row query tiles over the key tiles; cross: 128-row key tiles
    // over 128-row query tiles (debug flag bit 128: the keys-on-M cross mode,
    // over 64-row query chunks)
    const bool cross_t = cross && (g_debug_flags & 128);
    const int srow = cross ? kTile : pma_rows_per_item();
    const int scol = cross && !cross_t ? kTile : cross ? pma_rows_per_item() : kTile;
    if ((e = sched_launch(ss, q_off, kv_off, p->B, p->total_q, p->total_kv, srow, scol, p->mask, a.window,
                          cross ? 1 : 0, a.status, st)) != cudaSuccess ||
        (e = sched_launch(qs, q_off, kv_off, p->B, p->total_q, p->total_kv, kTile, kTile, p->mask, a.window, 0,
                          a.status, st)) != cudaSuccess ||
        (e = sched_launch(kv, q_off, kv_off, p->B, p->total_q, p->total_kv, kTile, kTile, p->mask, a.window, 1,
                          a.status, st)) != cudaSuccess)
      return cuda_fail("schedule launch", e);
    int* gate = reinterpret_cast<int*>(base + L.gate);
    if ((e = launch_pma_gate(q_off, kv_off, p->B, cross, gate, qs.n_tiles, kv.n_tiles, st)) != cudaSuccess)
      return cuda_fail("short-query gate launch", e);
    CUtensorMap sq_q, sq_do;
    if (make_map(&sq_q, q, p->total_q, p->H, p->D, pma_rows_per_item()) ||
        make_map(&sq_do, dout, p->total_q, p->H, p->D, pma_rows_per_item()))
      return cuda_fail("cuTensorMapEncodeTiled", cudaErrorInvalidValue);
    AttnArgs b = a;
    b.tiles = ss.sorted;
    b.n_tiles = ss.n_tiles;
    b.out0 = reinterpret_cast<__nv_bfloat16*>(dq);
    b.out1 = reinterpret_cast<__nv_bfloat16*>(dv);
    b.out2 = reinterpret_cast<__nv_bfloat16*>(dk);
    b.out_v8 = aligned32(dk) && aligned32(dv);
    prof(2, st);
    if (cross && !cross_t)
      e = launch_skv_bwd(p->act, hilo_for(*p), mq, mk, mv, mdo, b, gate, grid_for(dev, L.tiles_s, p->H), st);
    else
      e = launch_pma_bwd(p->act, hilo_for(*p), cross, sq_q, mk, mv, sq_do, b, gate, grid_for(dev, L.tiles_s, p->H),
                         st);
    if (e != cudaSuccess) return cuda_fail("fused backward kernel launch", e);
    prof(3, st);
  }
  // The dQ pass runs first: for softmax it also writes Di, which the dK/dV pass reads.
  if (p->total_q > 0) {
    if (!sq && (e = sched_launch(qs, q_off, kv_off, p->B, p->total_q, p->total_kv, kTile, kTile, p->mask, a.window,
                                 0, a.status, st)) != cudaSuccess)
      return cuda_fail("query-tile schedule launch", e);
    a.tiles = qs.sorted;
    a.n_tiles = qs.n_tiles;
    a.out0 = reinterpret_cast<__nv_bfloat16*>(dq);
    a.out1 = nullptr;
    a.out_v8 = aligned32(dq);
    prof(4, st);
    if ((e = launch_bwd_dq(p->D, p->act, hilo_for(*p), dq_split_rings(*p), mq, mk, mv, mdo, mo, a,
                             grid_for(dev, L.tiles_q, p->H), st)) != cudaSuccess)
      return cuda_fail("dQ kernel launch", e);
    prof(5, st);
  }
  if (p->total_kv > 0) {
    if (!sq && (e = sched_launch(kv, q_off, kv_off, p->B, p->total_q, p->total_kv, kTile, kTile, p->mask, a.window,
                                 1, a.status, st)) != cudaSuccess)
      return cuda_fail("key-tile schedule launch", e);
    a.tiles = kv.sorted;
    a.n_tiles = kv.n_tiles;
    a.out0 = reinterpret_cast<__nv_bfloat16*>(dk);
    a.out1 = reinterpret_cast<__nv_bfloat16*>(dv);
    a.out_v8 = aligned32(dk) && aligned32(dv);
    if (!sq) prof(2, st);
    if ((e = launch_bwd_dkdv(p->D, p->act, hilo_for(*p), mq, mk, mv, mdo, a, grid_for(dev, L.tiles_kv, p->H), st)) !=
        cudaSuccess)
      return cuda_fail("dK/dV kernel launch", e);
    if (!sq) prof(3, st);
  }
  return JATTN_OK;
}

}  // namespace
}  // namespace jattn

int jattn_bwd(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint16_t* q,
              const uint16_t* k, const uint16_t* v, const uint16_t* o, const float* lse, const uint16_t* dout,
              uint16_t* dq, uint16_t* dk, uint16_t* dv, void* ws, size_t ws_bytes, void* stream) {
  return jattn::bwd_impl(p, q_off, kv_off, q, k, v, o, lse, dout, nullptr, nullptr, 0, dq, dk, dv, ws, ws_bytes,
                         stream);
}

int jattn_bwd_rope(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, const uint16_t* q,
                   const uint16_t* k, const uint16_t* v, const uint16_t* o, const float* lse, const uint16_t* dout,
                   const float* rope_cos, const float* rope_sin, int64_t rope_rows, uint16_t* dq, uint16_t* dk,
                   uint16_t* dv, void* ws, size_t ws_bytes, void* stream) {
  const int rc = jattn::check_rope(rope_cos, rope_sin, rope_rows);
  if (rc != JATTN_OK) return rc;
  return jattn::bwd_impl(p, q_off, kv_off, q, k, v, o, lse, dout, rope_cos, rope_sin, rope_rows, dq, dk, dv, ws,
                         ws_bytes, stream);
}

int jattn_bwd_rope_workspace_size(const jattn_params_t* p, int64_t rope_rows, size_t* bytes) {
  if (!bytes) return JATTN_ERR_INVALID;
  int rc = check_params(p);
  if (rc != JATTN_OK) return rc;
  if (rope_rows < 1 || rope_rows > INT32_MAX) return JATTN_ERR_INVALID;
  *bytes = jattn::layout_for(*p).total + jattn::rope_extra_bytes(p->D, rope_rows);
  return JATTN_OK;
}

int64_t jattn_mxfp8_scale_rows(int64_t B, int64_t total) {
  return (B < 0 || total < 0) ? 0 : total / 32 + B;
}

int jattn_mxfp8_quantize(int64_t B, int64_t total, int H, int D, const int64_t* off, const uint16_t* x,
                         uint8_t* codes, uint8_t* scales, int32_t* block_start, void* ws, size_t ws_bytes,
                         void* stream) {
  if (B < 1 || B > INT32_MAX || total < 0 || total > INT32_MAX || H < 1 || (D != 64 && D != 128)) return JATTN_ERR_INVALID;
  if (!off || !block_start || (total > 0 && (!x || !codes || !scales))) return JATTN_ERR_INVALID;
  if (!aligned16(x) || !aligned16(codes)) return JATTN_ERR_ALIGN;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 512) return JATTN_ERR_WORKSPACE;
  DeviceInfo dev;
  int rc;
  if ((rc = device_info(dev)) != JATTN_OK) return rc;
  clear_stale_error();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DevStatus* status = reinterpret_cast<DevStatus*>(ws);
  int* n_blocks = reinterpret_cast<int*>(static_cast<char*>(ws) + 256);
  cudaError_t e;
  if ((e = sched_prefix_launch(off, B, total, 32, block_start, n_blocks, status, st)) != cudaSuccess)
    return cuda_fail("row-block prefix launch", e);
  if ((e = launch_mx_quant(off, static_cast<int>(B), H, D, jattn_mxfp8_scale_rows(B, total), x, codes, scales,
                           block_start, n_blocks, st)) != cudaSuccess)
    return cuda_fail("MXFP8 quantize launch", e);
  return JATTN_OK;
}

int jattn_rope(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, int keys, int inverse,
               const uint16_t* x, uint16_t* y, const float* rope_cos, const float* rope_sin, int64_t rope_rows,
               void* ws, size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc != JATTN_OK) return rc;
  if ((rc = check_rope(rope_cos, rope_sin, rope_rows)) != JATTN_OK) return rc;
  if (!q_off || !kv_off || (keys != 0 && keys != 1) || (inverse != 0 && inverse != 1)) return JATTN_ERR_INVALID;
  const int64_t total = keys ? p->total_kv : p->total_q;
  if (total > 0 && (!x || !y)) return JATTN_ERR_INVALID;
  if (!aligned16(x) || !aligned16(y)) return JATTN_ERR_ALIGN;
  // only the status word at the start of the workspace is used
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256) return JATTN_ERR_WORKSPACE;
  DeviceInfo dev;
  if ((rc = device_info(dev)) != JATTN_OK) return rc;
  clear_stale_error();
  const cudaError_t e =
      launch_rope(keys ? kv_off : q_off, keys ? q_off : kv_off, static_cast<int>(p->B), keys, inverse, p->H, p->D,
                  total, x, y, rope_cos, rope_sin, static_cast<int>(rope_rows), reinterpret_cast<DevStatus*>(ws),
                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? JATTN_OK : cuda_fail("rotary kernel launch", e);
}

int jattn_schedule(const jattn_params_t* p, const int64_t* q_off, const int64_t* kv_off, int row_tile,
                   int col_tile, int transposed, int32_t* tiles, int64_t max_tiles, int32_t* n_tiles, void* ws,
                   size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc != JATTN_OK) return rc;
  if (row_tile < kTile || col_tile < 1 || !q_off || !kv_off || !tiles || !n_tiles) return JATTN_ERR_INVALID;
  if ((rc = check_ws(p, ws, ws_bytes)) != JATTN_OK) return rc;
  const int64_t need = sched_max_tiles(p->B, transposed ? p->total_kv : p->total_q, row_tile);
  if (max_tiles < need) return JATTN_ERR_INVALID;
  clear_stale_error();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Layout L = layout_for(*p);
  char* base = static_cast<char*>(ws);
  // The row_tile = 128 regions are the largest; a coarser tiling fits in them.
  const SchedView sv = sched_carve(base + (transposed ? L.sched_kv : L.sched_q), p->B,
                                   transposed ? L.tiles_kv : L.tiles_q);
  const int window = (p->mask & (JATTN_MASK_WINDOW | JATTN_MASK_BLOCK)) ? p->window : 0;
  if (sched_launch(sv, q_off, kv_off, p->B, p->total_q, p->total_kv, row_tile, col_tile, p->mask, window,
                   transposed ? 1 : 0, reinterpret_cast<DevStatus*>(base), st) != cudaSuccess)
    return JATTN_ERR_CUDA;
  if (cudaMemcpyAsync(tiles, sv.sorted, sizeof(int4) * need, cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(n_tiles, sv.n_tiles, sizeof(int), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return JATTN_ERR_CUDA;
  return JATTN_OK;
}

int jattn_get_status(void* ws, void* stream, int* device_status) {
  if (!ws || !device_status) return JATTN_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DevStatus h{};
  if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return JATTN_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return JATTN_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(DevStatus), st) != cudaSuccess) return JATTN_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return JATTN_ERR_CUDA;
  *device_status = h.code;
  return JATTN_OK;
}

const char* jattn_error_string(int code) {
  switch (code) {
    case JATTN_OK: return "ok";
    case JATTN_ERR_INVALID: return "invalid argument";
    case JATTN_ERR_CUDA: return "CUDA runtime error";
    case JATTN_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case JATTN_ERR_ALIGN: return "value tensor not 16-byte aligned";
    case JATTN_ERR_OFFSETS: return "offsets are not a valid prefix sum of the row totals";
    case JATTN_ERR_TIMEOUT: return "a bounded pipeline wait expired";
    case JATTN_ERR_UNSUPPORTED: return "device is not sm_103";
    case JATTN_ERR_TOO_LARGE: return "problem needs more scratch than the allocation-free entry point holds";
    case JATTN_ERR_ROPE: return "a rotary position lies at or beyond the cos/sin tables' rows";
    default: return "unknown error code";
  }
}

const char* jattn_last_error(void) { return g_last_error; }

void jattn_profile_events(void* const* events) {
  for (int i = 0; i < 6; ++i) g_prof[i] = events ? static_cast<cudaEvent_t>(events[i]) : nullptr;
}

void jattn_debug_set(int flags, uint64_t timeout_ns) {
  g_debug_flags = flags;
  g_timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;
}

}  // extern "C"
