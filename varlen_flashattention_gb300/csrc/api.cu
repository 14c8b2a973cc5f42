// C ABI of the jagged FlashAttention library: argument validation, workspace
// layout, TMA descriptor encoding and kernel launches. See include/jfa.h for
// the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "jfa_internal.h"
#include "trace.cuh"

namespace jfa {

namespace {

// ------------------------------------------------------------------ helpers

bool aligned(const void* p, size_t a) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

uint64_t wait_budget_ns() {
  static std::atomic<uint64_t> cached{0};
  uint64_t v = cached.load(std::memory_order_relaxed);
  if (v) return v;
  double ms = 2000.0;
  if (const char* e = std::getenv("JFA_WAIT_BUDGET_MS")) {
    const double x = std::atof(e);
    if (x > 0) ms = x;
  }
  v = static_cast<uint64_t>(ms * 1e6);
  cached.store(v, std::memory_order_relaxed);
  return v;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::atomic<int> cache[64];
  if (dev >= 0 && dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D byte view [rows, cols] (e4m3 tiles) read in 128-row x 128-byte boxes
// with the 128-byte swizzle.
bool make_tmap_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  if (rows == 0) rows = 1;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(kTile)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 view [rows, cols] (cols contiguous) read in 128-row x 64-column
// boxes with the 128-byte swizzle the tcgen05 descriptors expect.
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows = kTile) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  if (rows == 0) rows = 1;  // nothing is read from an empty tensor; the map must still be valid
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows, cols] accumulator read and reduced in 32-column x 128-row boxes
// (128 bytes wide) with the 128-byte swizzle.
bool make_tmap_f32_acc(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  if (rows == 0) rows = 1;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kTile)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool good_dim(int d) { return d == 64 || d == 128 || d == 192; }

// Which forward kernel runs: head_dim 128 takes the flat-stream kernel, 64
// and 192 the per-tile kernel.
bool fwd_stream_path(int head_dim) { return head_dim == 128; }

jfa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? JFA_OK : JFA_ERR_CUDA; }

void record(void* events, int which, cudaStream_t s) {
  if (events) cudaEventRecord(static_cast<cudaEvent_t*>(events)[which], s);
}

// The optional event pair must hold two created events.
bool events_ok(void* events) {
  if (!events) return true;
  const cudaEvent_t* e = static_cast<const cudaEvent_t*>(events);
  return e[0] != nullptr && e[1] != nullptr;
}

// ------------------------------------------------------------------ workspace layouts

struct Layout {
  size_t status = 0, tile_base = 0, items = 0, item_seq = 0, lse2p = 0, deltap = 0, dq_acc = 0, part_o = 0,
         part_lse = 0;
  size_t bytes = 0;
  int64_t max_items = 0, pad_tiles = 0;
};

Layout self_layout(int64_t batch, int64_t heads, int64_t total, int64_t head_dim, bool bwd) {
  Layout L;
  size_t off = kStatusBytes;
  L.tile_base = off;
  off = align_up(off + 4 * (batch + 1), 256);
  L.pad_tiles = max_tiles(total, batch);
  L.max_items = heads * L.pad_tiles;
  L.items = off;
  off = align_up(off + 16 * L.max_items, 256);
  L.item_seq = off;
  off = align_up(off + 16 * L.max_items, 256);
  if (bwd) {
    L.lse2p = off;
    off = align_up(off + 4 * heads * L.pad_tiles * kTile, 256);
    L.deltap = off;
    off = align_up(off + 4 * heads * L.pad_tiles * kTile, 256);
    L.dq_acc = off;
    off = align_up(off + 4 * total * heads * head_dim, 256);
  }
  L.bytes = off;
  return L;
}

Layout bcast_layout(int64_t batch, int64_t q_len, int64_t heads, int64_t total_k, int64_t head_dim, bool bwd) {
  Layout L;
  size_t off = kStatusBytes;
  L.tile_base = off;
  off = align_up(off + 4 * (batch + 1), 256);
  const int64_t nqt = (q_len + kTile - 1) / kTile;
  L.max_items = bwd ? heads * max_tiles(total_k, batch) : batch * heads * nqt;
  L.items = off;
  off = align_up(off + 16 * L.max_items, 256);
  L.item_seq = off;
  off = align_up(off + 16 * L.max_items, 256);
  if (bwd) {
    L.pad_tiles = batch * nqt;
    L.lse2p = off;
    off = align_up(off + 4 * batch * heads * nqt * kTile, 256);
    L.deltap = off;
    off = align_up(off + 4 * batch * heads * nqt * kTile, 256);
    L.dq_acc = off;
    off = align_up(off + 4 * q_len * heads * head_dim, 256);
  }
  L.bytes = off;
  return L;
}

// Varlen / GQA: items are query tiles of every query head (forward) or key
// tiles of every KV head (backward); the padded LSE / delta rows and the dQ
// accumulator follow the queries.
Layout var_layout(int64_t batch, int64_t q_heads, int64_t kv_heads, int64_t total_q, int64_t total_k,
                  int64_t head_dim, bool bwd) {
  Layout L;
  size_t off = kStatusBytes;
  L.tile_base = off;
  off = align_up(off + 4 * (batch + 1), 256);
  L.pad_tiles = max_tiles(total_q, batch);
  L.max_items = bwd ? kv_heads * max_tiles(total_k, batch) : q_heads * L.pad_tiles;
  L.items = off;
  off = align_up(off + 16 * L.max_items, 256);
  L.item_seq = off;
  off = align_up(off + 16 * L.max_items, 256);
  if (bwd) {
    L.lse2p = off;
    off = align_up(off + 4 * q_heads * L.pad_tiles * kTile, 256);
    L.deltap = off;
    off = align_up(off + 4 * q_heads * L.pad_tiles * kTile, 256);
    L.dq_acc = off;
    off = align_up(off + 4 * total_q * q_heads * head_dim, 256);
  }
  L.bytes = off;
  return L;
}

// FP8 forward: the self-attention forward layout plus the transposed V blocks
// (one [128 x 128] byte block per key tile and head) unless the caller brings them.
Layout fp8_layout(int64_t batch, int64_t heads, int64_t total, size_t* vt_off, bool own_vt = true) {
  Layout L = self_layout(batch, heads, total, 128, false);
  *vt_off = L.bytes;
  if (own_vt) L.bytes = align_up(L.bytes + static_cast<size_t>(L.pad_tiles) * heads * 128 * 128, 256);
  return L;
}

// Small-query decode: the split partials of every (sequence, token, head) row.
Layout smallq_layout(int64_t batch, int64_t q_len, int64_t q_heads, int64_t splits) {
  Layout L;
  size_t off = kStatusBytes;
  L.part_o = off;
  off = align_up(off + 4 * splits * batch * q_len * q_heads * 128, 256);
  L.part_lse = off;
  off = align_up(off + 4 * splits * batch * q_len * q_heads, 256);
  L.bytes = off;
  return L;
}

Layout decode_layout(int64_t batch, int64_t q_heads, int64_t splits) {
  Layout L;
  size_t off = kStatusBytes;
  L.part_o = off;
  off = align_up(off + 4 * splits * batch * q_heads * 128, 256);
  L.part_lse = off;
  off = align_up(off + 4 * splits * batch * q_heads, 256);
  L.bytes = off;
  return L;
}

// ------------------------------------------------------------------ validation

jfa_status check_fwd(const jfa_fwd_args* a) {
  if (!a) return JFA_ERR_INVALID_ARG;
  if (a->batch < 0 || a->heads < 1 || a->total < 0 || a->max_seqlen < 0) return JFA_ERR_INVALID_ARG;
  if (!good_dim(a->head_dim)) return JFA_ERR_UNSUPPORTED;
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return JFA_ERR_INVALID_ARG;
  if (a->causal != 0 && a->causal != 1) return JFA_ERR_INVALID_ARG;
  if (!aligned(a->offsets, 4)) return JFA_ERR_INVALID_ARG;
  if (a->total > 0) {
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->o, 16) ||
        !aligned(a->lse, 4))
      return JFA_ERR_INVALID_ARG;
  }
  if (static_cast<int64_t>(a->total) * a->heads * a->head_dim >= (int64_t(1) << 40)) return JFA_ERR_INVALID_ARG;
  return JFA_OK;
}

jfa_status check_bwd(const jfa_bwd_args* a, int* chunk) {
  if (!a) return JFA_ERR_INVALID_ARG;
  if (a->batch < 0 || a->heads < 1 || a->total < 0 || a->max_seqlen < 0) return JFA_ERR_INVALID_ARG;
  if (!good_dim(a->head_dim)) return JFA_ERR_UNSUPPORTED;
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return JFA_ERR_INVALID_ARG;
  if (a->causal != 0 && a->causal != 1) return JFA_ERR_INVALID_ARG;
  int c = a->head_chunk;
  if (c == 0 && a->head_dim != 192) c = a->head_dim;  // head_dim 192: 0 stays "two passes"
  const bool ok_chunk =
      (c == 0) || (c == a->head_dim && a->head_dim != 192) || (c == 64 && a->head_dim >= 128);
  if (!ok_chunk) return JFA_ERR_UNSUPPORTED;  // head_dim 192 unchunked would overflow TMEM
  *chunk = c;
  if (!aligned(a->offsets, 4)) return JFA_ERR_INVALID_ARG;
  if (a->total > 0) {
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->o, 16) ||
        !aligned(a->dout, 16) || !aligned(a->lse, 4) || !aligned(a->dq, 16) || !aligned(a->dk, 16) ||
        !aligned(a->dv, 16))
      return JFA_ERR_INVALID_ARG;
  }
  if (static_cast<int64_t>(a->total) * a->heads * a->head_dim >= (int64_t(1) << 40)) return JFA_ERR_INVALID_ARG;
  return JFA_OK;
}

// Shared checks of the varlen entry points (the pointers are checked by the callers).
jfa_status check_var_common(int batch, int q_heads, int kv_heads, int head_dim, int max_q, int max_k, int total_q,
                            int total_k, float scale, int causal, const int32_t* q_offsets, const int32_t* k_offsets,
                            bool bwd) {
  if (batch < 0 || q_heads < 1 || kv_heads < 1 || max_q < 0 || max_k < 0 || total_q < 0 || total_k < 0)
    return JFA_ERR_INVALID_ARG;
  if (q_heads % kv_heads != 0) return JFA_ERR_INVALID_ARG;
  if (!good_dim(head_dim)) return JFA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return JFA_ERR_INVALID_ARG;
  if (!aligned(q_offsets, 4) || !aligned(k_offsets, 4)) return JFA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(total_q) * q_heads * head_dim >= (int64_t(1) << 40) ||
      static_cast<int64_t>(total_k) * kv_heads * head_dim >= (int64_t(1) << 40))
    return JFA_ERR_INVALID_ARG;
  // the queue's largest cost bucket: key tiles (forward), group x query tiles (backward)
  const int64_t kmax = bwd ? static_cast<int64_t>(q_heads / kv_heads) * ((max_q + kTile - 1) / kTile)
                           : (static_cast<int64_t>(max_k) + kTile - 1) / kTile;
  if (kmax > 32 * 1024) return JFA_ERR_UNSUPPORTED;
  return JFA_OK;
}

jfa_status check_bcast_common(int batch, int q_len, int heads, int head_dim, int max_seqlen_k, int total_k,
                              float scale) {
  if (batch < 0 || q_len < 0 || heads < 1 || max_seqlen_k < 0 || total_k < 0) return JFA_ERR_INVALID_ARG;
  if (!good_dim(head_dim)) return JFA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch) * q_len >= (int64_t(1) << 31)) return JFA_ERR_INVALID_ARG;
  return JFA_OK;
}

// The main backward launch(es). chunk 0 (head_dim 192 only) runs two passes
// over the head dimension, columns 0-127 and then 128-191: TMEM holds S^T and
// dP^T (256 columns) plus dV and dK slices of at most 128 columns each, and
// every pass rebuilds S^T and dP^T, so two passes do less work than three
// 64-wide ones. Otherwise each item is split into head_dim / chunk slices.
cudaError_t run_bwd_main(BwdLaunch bl, int chunk, int sms, int64_t max_items, const CUtensorMap& tq,
                         const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                         const CUtensorMap& tdk, const CUtensorMap& tdv, cudaStream_t stream) {
  const int64_t items = std::max<int64_t>(max_items, 1);
  if (chunk == 0) {
    bl.n_chunks = 1;
    bl.grid = static_cast<int>(std::min<int64_t>(sms, items));
    bl.head_chunk = 128;
    bl.col0 = 0;
    const cudaError_t e = launch_bwd_main(bl, tq, tk, tv, tdo, tdq, tdk, tdv, stream);
    if (e != cudaSuccess) return e;
    bl.head_chunk = 64;
    bl.col0 = 128;
    return launch_bwd_main(bl, tq, tk, tv, tdo, tdq, tdk, tdv, stream);
  }
  bl.head_chunk = chunk;
  bl.col0 = 0;
  bl.n_chunks = bl.head_dim / chunk;
  bl.grid = static_cast<int>(std::min<int64_t>(sms, items * bl.n_chunks));
  return launch_bwd_main(bl, tq, tk, tv, tdo, tdq, tdk, tdv, stream);
}

}  // namespace

// Scalar and pointer checks of the one-token paged decode (shared with the
// allocation-free entry point, which runs them before its scratch-size check).
jfa_status check_decode_args(const jfa_decode_args* a) {
  if (!a) return JFA_ERR_INVALID_ARG;
  if (a->batch < 0 || a->q_heads < 1 || a->kv_heads < 1 || a->page_size < 1 || a->num_pages < 0 ||
      a->max_pages < 0 || a->num_splits < 1 || a->num_splits > 128)
    return JFA_ERR_INVALID_ARG;
  if (a->q_heads % a->kv_heads != 0) return JFA_ERR_INVALID_ARG;
  const int g = a->q_heads / a->kv_heads;
  if (a->head_dim != 128 || !(g == 1 || g == 2 || g == 4 || g == 8 || g == 16)) return JFA_ERR_UNSUPPORTED;
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return JFA_ERR_INVALID_ARG;
  if (a->batch > 0) {
    if (!aligned(a->q, 16) || !aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) || !aligned(a->o, 16) ||
        !aligned(a->lse, 4) || !aligned(a->page_table, 4) || !aligned(a->seqlens_k, 4))
      return JFA_ERR_INVALID_ARG;
    if (a->split_bounds_out && !aligned(a->split_bounds_out, 4)) return JFA_ERR_INVALID_ARG;
  }
  if (static_cast<int64_t>(a->max_pages) * a->page_size >= (int64_t(1) << 31)) return JFA_ERR_INVALID_ARG;
  return JFA_OK;
}

}  // namespace jfa

using namespace jfa;

// ====================================================================== C ABI

extern "C" {

int32_t jfa_version(void) { return 100; }

const char* jfa_status_string(jfa_status s) {
  switch (s) {
    case JFA_OK: return "ok";
    case JFA_ERR_INVALID_ARG: return "invalid argument";
    case JFA_ERR_UNSUPPORTED: return "unsupported configuration";
    case JFA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case JFA_ERR_CUDA: return "CUDA error";
    case JFA_ERR_TIMEOUT: return "device pipeline wait timed out";
    case JFA_ERR_BAD_INPUT: return "inconsistent device input (offsets or page table)";
  }
  return "unknown status";
}

size_t jfa_fwd_workspace_size(const jfa_fwd_args* a) {
  if (!a) return 0;
  return self_layout(a->batch, a->heads, a->total, a->head_dim, false).bytes;
}

size_t jfa_bwd_workspace_size(const jfa_bwd_args* a) {
  if (!a) return 0;
  return self_layout(a->batch, a->heads, a->total, a->head_dim, true).bytes;
}

size_t jfa_bcast_fwd_workspace_size(const jfa_bcast_fwd_args* a) {
  if (!a) return 0;
  return bcast_layout(a->batch, a->q_len, a->heads, a->total_k, a->head_dim, false).bytes;
}

size_t jfa_bcast_bwd_workspace_size(const jfa_bcast_bwd_args* a) {
  if (!a) return 0;
  return bcast_layout(a->batch, a->q_len, a->heads, a->total_k, a->head_dim, true).bytes;
}

size_t jfa_decode_workspace_size(const jfa_decode_args* a) {
  if (!a) return 0;
  return decode_layout(a->batch, a->q_heads, a->num_splits).bytes;
}

jfa_status jfa_fwd(const jfa_fwd_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  jfa_status st = check_fwd(a);
  if (st != JFA_OK) return st;
  const Layout L = self_layout(a->batch, a->heads, a->total, a->head_dim, false);
  if (!aligned(ws, 256) || !events_ok(a->main_kernel_events)) return JFA_ERR_INVALID_ARG;
  if (ws_bytes < L.bytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  if (launch_status_clear(reinterpret_cast<int32_t*>(w), stream) != cudaSuccess) return JFA_ERR_CUDA;
  if (a->batch == 0 || a->total == 0) return JFA_OK;
  const int sms = sm_count();
  if (sms <= 0) return JFA_ERR_CUDA;
  CUtensorMap tq, tk, tv;
  const uint64_t cols = static_cast<uint64_t>(a->heads) * a->head_dim;
  if (!make_tmap_bf16(&tq, a->q, a->total, cols) || !make_tmap_bf16(&tk, a->k, a->total, cols) ||
      !make_tmap_bf16(&tv, a->v, a->total, cols))
    return JFA_ERR_CUDA;
  QueueParams qp{};
  qp.offsets = a->offsets;
  qp.batch = a->batch;
  qp.heads = a->heads;
  qp.total = a->total;
  qp.max_seqlen = a->max_seqlen;
  qp.causal = a->causal;
  qp.mode = kQueueSelfFwd;
  qp.q_len = 0;
  qp.status = status;
  qp.tile_base = reinterpret_cast<int32_t*>(w + L.tile_base);
  qp.items = reinterpret_cast<int4*>(w + L.items);
  qp.item_seq = reinterpret_cast<int4*>(w + L.item_seq);
  qp.max_items = static_cast<int32_t>(L.max_items);
  qp.count_index = 2;
  if (launch_queue(qp, stream) != cudaSuccess) return JFA_ERR_CUDA;
  cudaError_t e;
  const int grid = static_cast<int>(std::min<int64_t>(sms, std::max<int64_t>(L.max_items, 1)));
  record(a->main_kernel_events, 0, stream);
  if (fwd_stream_path(a->head_dim)) {
    CUtensorMap to;
    if (!make_tmap_bf16(&to, a->o, a->total, cols)) return JFA_ERR_CUDA;
    e = launch_fwd_stream(a->causal != 0, tq, tk, tv, to, qp.items, qp.item_seq, VarInfo{}, status, a->o, a->lse,
                          a->heads, a->total, 0, 0, a->scale, wait_budget_ns(), grid, stream);
  } else {
    e = launch_fwd(a->head_dim, a->causal != 0, tq, tk, tv, a->offsets, qp.items, qp.item_seq, VarInfo{}, status,
                   a->o, a->lse, a->heads, a->total, 0, 0, a->scale, wait_budget_ns(), grid, stream);
  }
  record(a->main_kernel_events, 1, stream);
  return cuda_status(e);
}

jfa_status jfa_bwd(const jfa_bwd_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int chunk = 0;
  jfa_status st = check_bwd(a, &chunk);
  if (st != JFA_OK) return st;
  const Layout L = self_layout(a->batch, a->heads, a->total, a->head_dim, true);
  if (!aligned(ws, 256) || !events_ok(a->main_kernel_events)) return JFA_ERR_INVALID_ARG;
  if (ws_bytes < L.bytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  if (launch_status_clear(reinterpret_cast<int32_t*>(w), stream) != cudaSuccess) return JFA_ERR_CUDA;
  if (a->batch == 0 || a->total == 0) return JFA_OK;
  const int sms = sm_count();
  if (sms <= 0) return JFA_ERR_CUDA;
  const int64_t n_acc = static_cast<int64_t>(a->total) * a->heads * a->head_dim;
  float* dq_acc = reinterpret_cast<float*>(w + L.dq_acc);  // zeroed by the pre-pass
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t cols = static_cast<uint64_t>(a->heads) * a->head_dim;
  if (!make_tmap_bf16(&tq, a->q, a->total, cols) || !make_tmap_bf16(&tk, a->k, a->total, cols) ||
      !make_tmap_bf16(&tv, a->v, a->total, cols) || !make_tmap_bf16(&tdo, a->dout, a->total, cols))
    return JFA_ERR_CUDA;
  QueueParams qp{};
  qp.offsets = a->offsets;
  qp.batch = a->batch;
  qp.heads = a->heads;
  qp.total = a->total;
  qp.max_seqlen = a->max_seqlen;
  qp.causal = a->causal;
  qp.mode = kQueueSelfBwd;
  qp.q_len = 0;
  qp.status = status;
  qp.tile_base = reinterpret_cast<int32_t*>(w + L.tile_base);
  qp.items = reinterpret_cast<int4*>(w + L.items);
  qp.item_seq = reinterpret_cast<int4*>(w + L.item_seq);
  qp.max_items = static_cast<int32_t>(L.max_items);
  qp.count_index = 2;
  if (launch_queue(qp, stream) != cudaSuccess) return JFA_ERR_CUDA;
  float* lse2p = reinterpret_cast<float*>(w + L.lse2p);
  float* deltap = reinterpret_cast<float*>(w + L.deltap);
  if (launch_bwd_pre(a->head_dim, a->o, a->dout, a->lse, a->offsets, qp.tile_base, status, a->batch, a->heads,
                     a->total, 0, 0, static_cast<int>(L.pad_tiles), static_cast<int>(L.pad_tiles), lse2p, deltap,
                     dq_acc, stream) != cudaSuccess)
    return JFA_ERR_CUDA;
  BwdLaunch bl{};
  bl.head_dim = a->head_dim;
  bl.head_chunk = chunk;
  bl.offsets = a->offsets;
  bl.tile_base = qp.tile_base;
  bl.items = qp.items;
  bl.item_seq = qp.item_seq;
  bl.status = status;
  bl.lse2p = lse2p;
  bl.deltap = deltap;
  bl.dq_acc = dq_acc;
  bl.dk = a->dk;
  bl.dv = a->dv;
  bl.heads = a->heads;
  bl.total = a->total;
  bl.bcast = 0;
  bl.q_len = 0;
  bl.causal = a->causal;
  bl.pad_tiles = static_cast<int>(L.pad_tiles);
  bl.scale = a->scale;
  bl.budget_ns = wait_budget_ns();
  record(a->main_kernel_events, 0, stream);
  CUtensorMap tdq, tdk, tdv;
  if (!make_tmap_f32_acc(&tdq, dq_acc, a->total, cols) || !make_tmap_bf16(&tdk, a->dk, a->total, cols) ||
      !make_tmap_bf16(&tdv, a->dv, a->total, cols))
    return JFA_ERR_CUDA;
  cudaError_t e = run_bwd_main(bl, chunk, sms, L.max_items, tq, tk, tv, tdo, tdq, tdk, tdv, stream);
  record(a->main_kernel_events, 1, stream);
  if (e != cudaSuccess) return JFA_ERR_CUDA;
  return cuda_status(launch_bwd_post(dq_acc, a->dq, n_acc, a->scale, status, sms, stream));
}

jfa_status jfa_fwd_broadcast_q(const jfa_bcast_fwd_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!a) return JFA_ERR_INVALID_ARG;
  jfa_status st = check_bcast_common(a->batch, a->q_len, a->heads, a->head_dim, a->max_seqlen_k, a->total_k, a->scale);
  if (st != JFA_OK) return st;
  if (!aligned(a->kv_offsets, 4)) return JFA_ERR_INVALID_ARG;
  if (a->batch > 0 && a->q_len > 0) {
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->o, 16) || !aligned(a->lse, 4))
      return JFA_ERR_INVALID_ARG;
  }
  const Layout L = bcast_layout(a->batch, a->q_len, a->heads, a->total_k, a->head_dim, false);
  if (!aligned(ws, 256) || !events_ok(a->main_kernel_events)) return JFA_ERR_INVALID_ARG;
  if (ws_bytes < L.bytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  if (launch_status_clear(reinterpret_cast<int32_t*>(w), stream) != cudaSuccess) return JFA_ERR_CUDA;
  if (a->batch == 0 || a->q_len == 0) return JFA_OK;
  const int sms = sm_count();
  if (sms <= 0) return JFA_ERR_CUDA;
  CUtensorMap tq, tk, tv;
  const uint64_t cols = static_cast<uint64_t>(a->heads) * a->head_dim;
  if (!make_tmap_bf16(&tq, a->q, a->q_len, cols) || !make_tmap_bf16(&tk, a->k, a->total_k, cols) ||
      !make_tmap_bf16(&tv, a->v, a->total_k, cols))
    return JFA_ERR_CUDA;
  QueueParams qp{};
  qp.offsets = a->kv_offsets;
  qp.batch = a->batch;
  qp.heads = a->heads;
  qp.total = a->total_k;
  qp.max_seqlen = a->max_seqlen_k;
  qp.causal = 0;
  qp.mode = kQueueBcastFwd;
  qp.q_len = a->q_len;
  qp.status = status;
  qp.tile_base = reinterpret_cast<int32_t*>(w + L.tile_base);
  qp.items = reinterpret_cast<int4*>(w + L.items);
  qp.item_seq = reinterpret_cast<int4*>(w + L.item_seq);
  qp.max_items = static_cast<int32_t>(L.max_items);
  qp.count_index = 2;
  if (launch_queue(qp, stream) != cudaSuccess) return JFA_ERR_CUDA;
  cudaError_t e;
  const int grid = static_cast<int>(std::min<int64_t>(sms, std::max<int64_t>(L.max_items, 1)));
  record(a->main_kernel_events, 0, stream);
  if (fwd_stream_path(a->head_dim)) {
    CUtensorMap to;
    if (!make_tmap_bf16(&to, a->o, static_cast<uint64_t>(a->batch) * a->q_len, cols)) return JFA_ERR_CUDA;
    e = launch_fwd_stream(false, tq, tk, tv, to, qp.items, qp.item_seq, VarInfo{}, status, a->o, a->lse, a->heads,
                          a->total_k, 1, a->q_len, a->scale, wait_budget_ns(), grid, stream);
  } else {
    e = launch_fwd(a->head_dim, false, tq, tk, tv, a->kv_offsets, qp.items, qp.item_seq, VarInfo{}, status, a->o,
                   a->lse, a->heads, a->total_k, 1, a->q_len, a->scale, wait_budget_ns(), grid, stream);
  }
  record(a->main_kernel_events, 1, stream);
  return cuda_status(e);
}

jfa_status jfa_bwd_broadcast_q(const jfa_bcast_bwd_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!a) return JFA_ERR_INVALID_ARG;
  jfa_status st = check_bcast_common(a->batch, a->q_len, a->heads, a->head_dim, a->max_seqlen_k, a->total_k, a->scale);
  if (st != JFA_OK) return st;
  if (!aligned(a->kv_offsets, 4)) return JFA_ERR_INVALID_ARG;
  if (a->batch > 0 && a->q_len > 0) {
    if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->o, 16) ||
        !aligned(a->dout, 16) || !aligned(a->lse, 4) || !aligned(a->dq, 16) || !aligned(a->dk, 16) ||
        !aligned(a->dv, 16))
      return JFA_ERR_INVALID_ARG;
  }
  const Layout L = bcast_layout(a->batch, a->q_len, a->heads, a->total_k, a->head_dim, true);
  if (!aligned(ws, 256) || !events_ok(a->main_kernel_events)) return JFA_ERR_INVALID_ARG;
  if (ws_bytes < L.bytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  if (launch_status_clear(reinterpret_cast<int32_t*>(w), stream) != cudaSuccess) return JFA_ERR_CUDA;
  if (a->q_len == 0) return JFA_OK;
  const int64_t n_acc = static_cast<int64_t>(a->q_len) * a->heads * a->head_dim;
  float* dq_acc = reinterpret_cast<float*>(w + L.dq_acc);  // zeroed by the pre-pass when there are keys
  const int sms = sm_count();
  if (sms <= 0) return JFA_ERR_CUDA;
  if (!(a->batch > 0 && a->total_k > 0)) {
    if (cudaMemsetAsync(dq_acc, 0, 4 * n_acc, stream) != cudaSuccess) return JFA_ERR_CUDA;
  } else {
    CUtensorMap tq, tk, tv, tdo;
    const uint64_t cols = static_cast<uint64_t>(a->heads) * a->head_dim;
    if (!make_tmap_bf16(&tq, a->q, a->q_len, cols) || !make_tmap_bf16(&tk, a->k, a->total_k, cols) ||
        !make_tmap_bf16(&tv, a->v, a->total_k, cols) ||
        !make_tmap_bf16(&tdo, a->dout, static_cast<uint64_t>(a->batch) * a->q_len, cols))
      return JFA_ERR_CUDA;
    QueueParams qp{};
    qp.offsets = a->kv_offsets;
    qp.batch = a->batch;
    qp.heads = a->heads;
    qp.total = a->total_k;
    qp.max_seqlen = a->max_seqlen_k;
    qp.causal = 0;
    qp.mode = kQueueBcastBwd;
    qp.q_len = a->q_len;
    qp.status = status;
    qp.tile_base = reinterpret_cast<int32_t*>(w + L.tile_base);
    qp.items = reinterpret_cast<int4*>(w + L.items);
    qp.item_seq = reinterpret_cast<int4*>(w + L.item_seq);
    qp.max_items = static_cast<int32_t>(L.max_items);
    qp.count_index = 2;
    if (launch_queue(qp, stream) != cudaSuccess) return JFA_ERR_CUDA;
    float* lse2p = reinterpret_cast<float*>(w + L.lse2p);
    float* deltap = reinterpret_cast<float*>(w + L.deltap);
    if (launch_bwd_pre(a->head_dim, a->o, a->dout, a->lse, a->kv_offsets, nullptr, status, a->batch, a->heads,
                       a->total_k, 1, a->q_len, 0, static_cast<int>(L.pad_tiles), lse2p, deltap, dq_acc,
                       stream) != cudaSuccess)
      return JFA_ERR_CUDA;
    BwdLaunch bl{};
    bl.head_dim = a->head_dim;
    bl.offsets = a->kv_offsets;
    bl.tile_base = qp.tile_base;
    bl.items = qp.items;
    bl.item_seq = qp.item_seq;
    bl.status = status;
    bl.lse2p = lse2p;
    bl.deltap = deltap;
    bl.dq_acc = dq_acc;
    bl.dk = a->dk;
    bl.dv = a->dv;
    bl.heads = a->heads;
    bl.total = a->total_k;
    bl.bcast = 1;
    bl.q_len = a->q_len;
    bl.causal = 0;
    bl.pad_tiles = 0;
    bl.scale = a->scale;
    bl.budget_ns = wait_budget_ns();
    record(a->main_kernel_events, 0, stream);
    CUtensorMap tdq, tdk, tdv;
    if (!make_tmap_f32_acc(&tdq, dq_acc, a->q_len, cols) || !make_tmap_bf16(&tdk, a->dk, a->total_k, cols) ||
        !make_tmap_bf16(&tdv, a->dv, a->total_k, cols))
      return JFA_ERR_CUDA;
    // head_dim 192: the two head-axis passes of jfa_bwd; otherwise one slice
    const int chunk = a->head_dim == 192 ? 0 : a->head_dim;
    cudaError_t e = run_bwd_main(bl, chunk, sms, L.max_items, tq, tk, tv, tdo, tdq, tdk, tdv, stream);
    record(a->main_kernel_events, 1, stream);
    if (e != cudaSuccess) return JFA_ERR_CUDA;
  }
  return cuda_status(launch_bwd_post(dq_acc, a->dq, n_acc, a->scale, status, sms, stream));
}

jfa_status jfa_decode_splitkv(const jfa_decode_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const jfa_status st = check_decode_args(a);
  if (st != JFA_OK) return st;
  const Layout L = decode_layout(a->batch, a->q_heads, a->num_splits);
  if (!aligned(ws, 256) || !events_ok(a->main_kernel_events)) return JFA_ERR_INVALID_ARG;
  if (ws_bytes < L.bytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (launch_status_clear(reinterpret_cast<int32_t*>(w), stream) != cudaSuccess) return JFA_ERR_CUDA;
  if (a->batch == 0) return JFA_OK;
  return cuda_status(launch_decode(*a, reinterpret_cast<float*>(w + L.part_o), reinterpret_cast<float*>(w + L.part_lse),
                                   reinterpret_cast<int32_t*>(w), stream));
}

size_t jfa_varlen_fwd_workspace_size(const jfa_varlen_fwd_args* a) {
  if (!a) return 0;
  return var_layout(a->batch, a->q_heads, a->kv_heads, a->total_q, a->total_k, a->head_dim, false).bytes;
}

size_t jfa_varlen_bwd_workspace_size(const jfa_varlen_bwd_args* a) {
  if (!a) return 0;
  return var_layout(a->batch, a->q_heads, a->kv_heads, a->total_q, a->total_k, a->head_dim, true).bytes;
}

jfa_status jfa_fwd_varlen(const jfa_varlen_fwd_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!a) return JFA_ERR_INVALID_ARG;
  jfa_status st = check_var_common(a->batch, a->q_heads, a->kv_heads, a->head_dim, a->max_seqlen_q, a->max_seqlen_k,
                                   a->total_q, a->total_k, a->scale, a->causal, a->q_offsets, a->k_offsets, false);
  if (st != JFA_OK) return st;
  if (a->total_q > 0 && (!aligned(a->q, 16) || !aligned(a->o, 16) || !aligned(a->lse, 4))) return JFA_ERR_INVALID_ARG;
  if (a->total_k > 0 && (!aligned(a->k, 16) || !aligned(a->v, 16))) return JFA_ERR_INVALID_ARG;
  const Layout L = var_layout(a->batch, a->q_heads, a->kv_heads, a->total_q, a->total_k, a->head_dim, false);
  if (!aligned(ws, 256) || !events_ok(a->main_kernel_events)) return JFA_ERR_INVALID_ARG;
  if (ws_bytes < L.bytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  if (launch_status_clear(reinterpret_cast<int32_t*>(w), stream) != cudaSuccess) return JFA_ERR_CUDA;
  if (a->batch == 0 || a->total_q == 0) return JFA_OK;
  const int sms = sm_count();
  if (sms <= 0) return JFA_ERR_CUDA;
  // with no keys at all the K/V maps are never read; they still need a valid base
  const void* kb = a->total_k > 0 ? a->k : a->q;
  const void* vb = a->total_k > 0 ? a->v : a->q;
  CUtensorMap tq, tk, tv;
  const uint64_t qcols = static_cast<uint64_t>(a->q_heads) * a->head_dim;
  const uint64_t kcols = static_cast<uint64_t>(a->kv_heads) * a->head_dim;
  if (!make_tmap_bf16(&tq, a->q, a->total_q, qcols) || !make_tmap_bf16(&tk, kb, a->total_k, kcols) ||
      !make_tmap_bf16(&tv, vb, a->total_k, kcols))
    return JFA_ERR_CUDA;
  QueueParams qp{};
  qp.offsets = a->q_offsets;
  qp.k_offsets = a->k_offsets;
  qp.batch = a->batch;
  qp.heads = a->q_heads;
  qp.total = a->total_q;
  qp.max_seqlen = a->max_seqlen_q;
  qp.total_k = a->total_k;
  qp.max_seqlen_k = a->max_seqlen_k;
  qp.group = a->q_heads / a->kv_heads;
  qp.causal = a->causal;
  qp.mode = kQueueVarFwd;
  qp.status = status;
  qp.tile_base = reinterpret_cast<int32_t*>(w + L.tile_base);
  qp.items = reinterpret_cast<int4*>(w + L.items);
  qp.item_seq = reinterpret_cast<int4*>(w + L.item_seq);
  qp.max_items = static_cast<int32_t>(L.max_items);
  qp.count_index = 2;
  if (launch_queue(qp, stream) != cudaSuccess) return JFA_ERR_CUDA;
  VarInfo vi;
  vi.var = 1;
  vi.group = qp.group;
  cudaError_t e;
  const int grid = static_cast<int>(std::min<int64_t>(sms, std::max<int64_t>(L.max_items, 1)));
  record(a->main_kernel_events, 0, stream);
  if (fwd_stream_path(a->head_dim)) {
    CUtensorMap to;
    if (!make_tmap_bf16(&to, a->o, a->total_q, qcols)) return JFA_ERR_CUDA;
    e = launch_fwd_stream(a->causal != 0, tq, tk, tv, to, qp.items, qp.item_seq, vi, status, a->o, a->lse,
                          a->q_heads, a->total_q, 0, 0, a->scale, wait_budget_ns(), grid, stream);
  } else {
    e = launch_fwd(a->head_dim, a->causal != 0, tq, tk, tv, a->q_offsets, qp.items, qp.item_seq, vi, status, a->o,
                   a->lse, a->q_heads, a->total_q, 0, 0, a->scale, wait_budget_ns(), grid, stream);
  }
  record(a->main_kernel_events, 1, stream);
  return cuda_status(e);
}

jfa_status jfa_bwd_varlen(const jfa_varlen_bwd_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!a) return JFA_ERR_INVALID_ARG;
  jfa_status st = check_var_common(a->batch, a->q_heads, a->kv_heads, a->head_dim, a->max_seqlen_q, a->max_seqlen_k,
                                   a->total_q, a->total_k, a->scale, a->causal, a->q_offsets, a->k_offsets, true);
  if (st != JFA_OK) return st;
  int chunk = a->head_chunk;
  if (chunk == 0 && a->head_dim != 192) chunk = a->head_dim;  // head_dim 192: 0 stays "two passes"
  if (!(chunk == 0 || (chunk == a->head_dim && a->head_dim != 192) || (chunk == 64 && a->head_dim >= 128)))
    return JFA_ERR_UNSUPPORTED;  // head_dim 192 unchunked would overflow TMEM
  if (a->total_q > 0 && (!aligned(a->q, 16) || !aligned(a->o, 16) || !aligned(a->dout, 16) || !aligned(a->lse, 4) ||
                         !aligned(a->dq, 16)))
    return JFA_ERR_INVALID_ARG;
  if (a->total_k > 0 && (!aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->dk, 16) || !aligned(a->dv, 16)))
    return JFA_ERR_INVALID_ARG;
  const Layout L = var_layout(a->batch, a->q_heads, a->kv_heads, a->total_q, a->total_k, a->head_dim, true);
  if (!aligned(ws, 256) || !events_ok(a->main_kernel_events)) return JFA_ERR_INVALID_ARG;
  if (ws_bytes < L.bytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  if (launch_status_clear(reinterpret_cast<int32_t*>(w), stream) != cudaSuccess) return JFA_ERR_CUDA;
  const size_t kv_bytes = static_cast<size_t>(a->total_k) * a->kv_heads * a->head_dim * 2;
  if (a->batch == 0 || a->total_k == 0 || a->total_q == 0) {
    // no (query, key) pair anywhere: every gradient is zero
    if (kv_bytes && (cudaMemsetAsync(a->dk, 0, kv_bytes, stream) != cudaSuccess ||
                     cudaMemsetAsync(a->dv, 0, kv_bytes, stream) != cudaSuccess))
      return JFA_ERR_CUDA;
    const size_t q_bytes = static_cast<size_t>(a->total_q) * a->q_heads * a->head_dim * 2;
    if (q_bytes && cudaMemsetAsync(a->dq, 0, q_bytes, stream) != cudaSuccess) return JFA_ERR_CUDA;
    return JFA_OK;
  }
  const int sms = sm_count();
  if (sms <= 0) return JFA_ERR_CUDA;
  const int64_t n_acc = static_cast<int64_t>(a->total_q) * a->q_heads * a->head_dim;
  float* dq_acc = reinterpret_cast<float*>(w + L.dq_acc);  // zeroed by the pre-pass
  CUtensorMap tq, tk, tv, tdo;
  const uint64_t qcols = static_cast<uint64_t>(a->q_heads) * a->head_dim;
  const uint64_t kcols = static_cast<uint64_t>(a->kv_heads) * a->head_dim;
  if (!make_tmap_bf16(&tq, a->q, a->total_q, qcols) || !make_tmap_bf16(&tk, a->k, a->total_k, kcols) ||
      !make_tmap_bf16(&tv, a->v, a->total_k, kcols) || !make_tmap_bf16(&tdo, a->dout, a->total_q, qcols))
    return JFA_ERR_CUDA;
  QueueParams qp{};
  qp.offsets = a->q_offsets;
  qp.k_offsets = a->k_offsets;
  qp.batch = a->batch;
  qp.heads = a->kv_heads;
  qp.total = a->total_q;
  qp.max_seqlen = a->max_seqlen_q;
  qp.total_k = a->total_k;
  qp.max_seqlen_k = a->max_seqlen_k;
  qp.group = a->q_heads / a->kv_heads;
  qp.causal = a->causal;
  qp.mode = kQueueVarBwd;
  qp.status = status;
  qp.tile_base = reinterpret_cast<int32_t*>(w + L.tile_base);
  qp.items = reinterpret_cast<int4*>(w + L.items);
  qp.item_seq = reinterpret_cast<int4*>(w + L.item_seq);
  qp.max_items = static_cast<int32_t>(L.max_items);
  qp.count_index = 2;
  if (launch_queue(qp, stream) != cudaSuccess) return JFA_ERR_CUDA;
  float* lse2p = reinterpret_cast<float*>(w + L.lse2p);
  float* deltap = reinterpret_cast<float*>(w + L.deltap);
  if (launch_bwd_pre(a->head_dim, a->o, a->dout, a->lse, a->q_offsets, qp.tile_base, status, a->batch, a->q_heads,
                     a->total_q, 0, 0, static_cast<int>(L.pad_tiles), static_cast<int>(L.pad_tiles), lse2p, deltap,
                     dq_acc, stream) != cudaSuccess)
    return JFA_ERR_CUDA;
  BwdLaunch bl{};
  bl.head_dim = a->head_dim;
  bl.head_chunk = chunk;
  bl.offsets = a->q_offsets;
  bl.tile_base = qp.tile_base;
  bl.items = qp.items;
  bl.item_seq = qp.item_seq;
  bl.status = status;
  bl.lse2p = lse2p;
  bl.deltap = deltap;
  bl.dq_acc = dq_acc;
  bl.dk = a->dk;
  bl.dv = a->dv;
  bl.heads = a->q_heads;
  bl.total = a->total_q;
  bl.bcast = 0;
  bl.q_len = 0;
  bl.causal = a->causal;
  bl.pad_tiles = static_cast<int>(L.pad_tiles);
  bl.var = 1;
  bl.group = qp.group;
  bl.kv_heads = a->kv_heads;
  bl.scale = a->scale;
  bl.budget_ns = wait_budget_ns();
  CUtensorMap tdq, tdk, tdv;
  if (!make_tmap_f32_acc(&tdq, dq_acc, a->total_q, qcols) || !make_tmap_bf16(&tdk, a->dk, a->total_k, kcols) ||
      !make_tmap_bf16(&tdv, a->dv, a->total_k, kcols))
    return JFA_ERR_CUDA;
  record(a->main_kernel_events, 0, stream);
  cudaError_t e = run_bwd_main(bl, chunk, sms, L.max_items, tq, tk, tv, tdo, tdq, tdk, tdv, stream);
  record(a->main_kernel_events, 1, stream);
  if (e != cudaSuccess) return JFA_ERR_CUDA;
  return cuda_status(launch_bwd_post(dq_acc, a->dq, n_acc, a->scale, status, sms, stream));
}

size_t jfa_decode_smallq_workspace_size(const jfa_decode_smallq_args* a) {
  if (!a) return 0;
  return smallq_layout(a->batch, a->q_len, a->q_heads, a->num_splits).bytes;
}

jfa_status jfa_decode_smallq(const jfa_decode_smallq_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!a) return JFA_ERR_INVALID_ARG;
  if (a->batch < 0 || a->q_len < 1 || a->q_heads < 1 || a->kv_heads < 1 || a->page_size < 1 || a->num_pages < 0 ||
      a->max_pages < 0 || a->num_splits < 1 || a->num_splits > 128 || a->min_split_tokens < 0)
    return JFA_ERR_INVALID_ARG;
  if (a->q_heads % a->kv_heads != 0) return JFA_ERR_INVALID_ARG;
  const int g = a->q_heads / a->kv_heads;
  if (a->head_dim != 128 || !(g == 1 || g == 2 || g == 4 || g == 8 || g == 16)) return JFA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(g) * a->q_len > 16) return JFA_ERR_UNSUPPORTED;  // rows of one tile
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return JFA_ERR_INVALID_ARG;
  if (a->batch > 0) {
    if (!aligned(a->q, 16) || !aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) || !aligned(a->o, 16) ||
        !aligned(a->lse, 4) || !aligned(a->page_table, 4) || !aligned(a->seqlens_k, 4))
      return JFA_ERR_INVALID_ARG;
    if (a->split_bounds_out && !aligned(a->split_bounds_out, 4)) return JFA_ERR_INVALID_ARG;
    if (a->split_counts_out && !aligned(a->split_counts_out, 4)) return JFA_ERR_INVALID_ARG;
  }
  if (static_cast<int64_t>(a->max_pages) * a->page_size >= (int64_t(1) << 31)) return JFA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(a->batch) * a->q_len * a->q_heads >= (int64_t(1) << 31)) return JFA_ERR_INVALID_ARG;
  const Layout L = smallq_layout(a->batch, a->q_len, a->q_heads, a->num_splits);
  if (!aligned(ws, 256) || !events_ok(a->main_kernel_events)) return JFA_ERR_INVALID_ARG;
  if (ws_bytes < L.bytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (launch_status_clear(reinterpret_cast<int32_t*>(w), stream) != cudaSuccess) return JFA_ERR_CUDA;
  if (a->batch == 0) return JFA_OK;
  DecodeLaunch d;
  d.q = a->q;
  d.k_cache = a->k_cache;
  d.v_cache = a->v_cache;
  d.page_table = a->page_table;
  d.seqlens_k = a->seqlens_k;
  d.batch = a->batch;
  d.q_len = a->q_len;
  d.q_heads = a->q_heads;
  d.kv_heads = a->kv_heads;
  d.page_size = a->page_size;
  d.num_pages = a->num_pages;
  d.max_pages = a->max_pages;
  d.num_splits = a->num_splits;
  d.min_split_tokens = a->min_split_tokens;
  d.scale = a->scale;
  d.o = a->o;
  d.lse = a->lse;
  d.split_bounds_out = a->split_bounds_out;
  d.split_counts_out = a->split_counts_out;
  d.main_kernel_events = a->main_kernel_events;
  return cuda_status(launch_decode_general(d, reinterpret_cast<float*>(w + L.part_o),
                                           reinterpret_cast<float*>(w + L.part_lse), reinterpret_cast<int32_t*>(w),
                                           stream));
}

jfa_status jfa_selftest_wait_timeout(int32_t budget_us, void* ws, cudaStream_t stream) {
  if (budget_us < 1 || budget_us > 10 * 1000 * 1000 || !aligned(ws, 256)) return JFA_ERR_INVALID_ARG;
  if (cudaMemsetAsync(ws, 0, kStatusBytes, stream) != cudaSuccess) return JFA_ERR_CUDA;
  return cuda_status(launch_selftest_wait(static_cast<int32_t*>(ws), static_cast<uint64_t>(budget_us) * 1000, stream));
}

size_t jfa_fwd_fp8_workspace_size(const jfa_fwd_fp8_args* a) {
  if (!a) return 0;
  size_t vt_off = 0;
  return fp8_layout(a->batch, a->heads, a->total, &vt_off, a->vt == nullptr).bytes;
}

size_t jfa_fp8_vt_bytes(int32_t batch, int32_t heads, int32_t total) {
  if (batch < 0 || heads < 1 || total < 0) return 0;
  return static_cast<size_t>(max_tiles(total, batch)) * heads * 128 * 128;
}

size_t jfa_fp8_quantize_v_workspace_size(const jfa_fp8_quantize_v_args* a) {
  if (!a) return 0;
  return self_layout(a->batch, a->heads, a->total, 128, false).bytes;
}

jfa_status jfa_fp8_quantize_v(const jfa_fp8_quantize_v_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!a) return JFA_ERR_INVALID_ARG;
  if (a->batch < 0 || a->heads < 1 || a->total < 0 || a->max_seqlen < 0) return JFA_ERR_INVALID_ARG;
  if (a->head_dim != 128) return JFA_ERR_UNSUPPORTED;
  if (!(a->v_descale > 0.f) || !std::isfinite(a->v_descale)) return JFA_ERR_INVALID_ARG;
  const float inv = 1.0f / a->v_descale;
  if (!std::isfinite(inv) || !(inv > 0.f)) return JFA_ERR_INVALID_ARG;
  if (!aligned(a->offsets, 4)) return JFA_ERR_INVALID_ARG;
  if (a->total > 0 && (!aligned(a->v, 16) || !aligned(a->vt, 16))) return JFA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(a->total) * a->heads * 128 >= (int64_t(1) << 40)) return JFA_ERR_INVALID_ARG;
  const Layout L = self_layout(a->batch, a->heads, a->total, 128, false);
  if (!aligned(ws, 256)) return JFA_ERR_INVALID_ARG;
  if (ws_bytes < L.bytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  if (launch_status_clear(status, stream) != cudaSuccess) return JFA_ERR_CUDA;
  if (a->batch == 0 || a->total == 0) return JFA_OK;
  QueueParams qp{};  // every 128-key tile of every sequence and head, as the forward numbers them
  qp.offsets = a->offsets;
  qp.batch = a->batch;
  qp.heads = a->heads;
  qp.total = a->total;
  qp.max_seqlen = a->max_seqlen;
  qp.causal = 0;
  qp.mode = kQueueSelfFwd;
  qp.status = status;
  qp.tile_base = reinterpret_cast<int32_t*>(w + L.tile_base);
  qp.items = reinterpret_cast<int4*>(w + L.items);
  qp.item_seq = reinterpret_cast<int4*>(w + L.item_seq);
  qp.max_items = static_cast<int32_t>(L.max_items);
  qp.count_index = 2;
  if (launch_queue(qp, stream) != cudaSuccess) return JFA_ERR_CUDA;
  return cuda_status(launch_vt_transpose(a->v, qp.items, qp.item_seq, status, a->heads, static_cast<int>(L.max_items),
                                         a->vt, stream, &inv));
}

jfa_status jfa_fwd_fp8(const jfa_fwd_fp8_args* a, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!a) return JFA_ERR_INVALID_ARG;
  if (a->batch < 0 || a->heads < 1 || a->total < 0 || a->max_seqlen < 0) return JFA_ERR_INVALID_ARG;
  if (a->head_dim != 128) return JFA_ERR_UNSUPPORTED;
  if (!(a->scale > 0.f) || !std::isfinite(a->scale) || a->causal < 0 || a->causal > 1) return JFA_ERR_INVALID_ARG;
  for (float f : {a->q_descale, a->k_descale, a->v_descale})
    if (!(f > 0.f) || !std::isfinite(f)) return JFA_ERR_INVALID_ARG;
  if (!aligned(a->offsets, 4)) return JFA_ERR_INVALID_ARG;
  const bool own_vt = a->vt == nullptr;  // else the caller's blocks from jfa_fp8_quantize_v
  if (a->total > 0 && (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(own_vt ? a->v : a->vt, 16) ||
                       !aligned(a->o, 16) || !aligned(a->lse, 4)))
    return JFA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(a->total) * a->heads * 128 >= (int64_t(1) << 40)) return JFA_ERR_INVALID_ARG;
  size_t vt_off = 0;
  const Layout L = fp8_layout(a->batch, a->heads, a->total, &vt_off, own_vt);
  if (!aligned(ws, 256) || !events_ok(a->main_kernel_events)) return JFA_ERR_INVALID_ARG;
  if (ws_bytes < L.bytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  if (launch_status_clear(reinterpret_cast<int32_t*>(w), stream) != cudaSuccess) return JFA_ERR_CUDA;
  if (a->batch == 0 || a->total == 0) return JFA_OK;
  const int sms = sm_count();
  if (sms <= 0) return JFA_ERR_CUDA;
  QueueParams qp{};
  qp.offsets = a->offsets;
  qp.batch = a->batch;
  qp.heads = a->heads;
  qp.total = a->total;
  qp.max_seqlen = a->max_seqlen;
  qp.causal = a->causal;
  qp.mode = kQueueSelfFwd;
  qp.status = status;
  qp.tile_base = reinterpret_cast<int32_t*>(w + L.tile_base);
  qp.items = reinterpret_cast<int4*>(w + L.items);
  qp.item_seq = reinterpret_cast<int4*>(w + L.item_seq);
  qp.max_items = static_cast<int32_t>(L.max_items);
  qp.count_index = 2;
  if (launch_queue(qp, stream) != cudaSuccess) return JFA_ERR_CUDA;
  const void* vt = own_vt ? static_cast<const void*>(w + vt_off) : a->vt;
  if (own_vt && launch_vt_transpose(a->v, qp.items, qp.item_seq, status, a->heads, static_cast<int>(L.max_items),
                                    w + vt_off, stream) != cudaSuccess)
    return JFA_ERR_CUDA;
  CUtensorMap tq, tk, tvt;
  const uint64_t cols = static_cast<uint64_t>(a->heads) * 128;
  if (!make_tmap_u8(&tq, a->q, a->total, cols) || !make_tmap_u8(&tk, a->k, a->total, cols) ||
      !make_tmap_u8(&tvt, vt, static_cast<uint64_t>(L.pad_tiles) * a->heads * 128, 128))
    return JFA_ERR_CUDA;
  const int grid = static_cast<int>(std::min<int64_t>(sms, std::max<int64_t>(L.max_items, 1)));
  const float s_log2 = a->scale * a->q_descale * a->k_descale * 1.4426950408889634f;
  CUtensorMap to;
  if (!make_tmap_bf16(&to, a->o, a->total, cols)) return JFA_ERR_CUDA;
  record(a->main_kernel_events, 0, stream);
  const cudaError_t e = launch_fwd_fp8(a->causal != 0, tq, tk, tvt, to, qp.items, qp.item_seq, status, a->o, a->lse,
                                       a->heads, a->total, s_log2, a->v_descale, wait_budget_ns(), grid, stream);
  record(a->main_kernel_events, 1, stream);
  return cuda_status(e);
}

int32_t jfa_trace_compiled(void) {
#ifdef JFA_TRACE
  return 1;
#else
  return 0;
#endif
}

jfa_status jfa_trace_enable(void* buffer, size_t bytes, int32_t records_per_warp) {
#ifdef JFA_TRACE
  if (buffer == nullptr) {
    jfa::set_trace_buffer(nullptr, 0, 0);
    return JFA_OK;
  }
  if (records_per_warp < 1 || !aligned(buffer, 16)) return JFA_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return JFA_ERR_CUDA;
  const size_t need = static_cast<size_t>(sms) * jfa::trace::kWarpSlots * static_cast<size_t>(records_per_warp) *
                      jfa::trace::kRecordBytes;
  if (bytes < need) return JFA_ERR_INVALID_ARG;
  jfa::set_trace_buffer(buffer, records_per_warp, sms);
  return JFA_OK;
#else
  (void)buffer;
  (void)bytes;
  (void)records_per_warp;
  return JFA_ERR_UNSUPPORTED;
#endif
}

jfa_status jfa_read_device_status(const void* ws, cudaStream_t stream, int32_t* detail) {
  if (!aligned(ws, 4)) return JFA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return JFA_ERR_CUDA;
  int32_t h[2] = {0, 0};
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return JFA_ERR_CUDA;
  if (detail) *detail = h[1];
  return static_cast<jfa_status>(h[0]);
}

}  // extern "C"
