// Internal definitions shared by the host layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

#include "../../include/jfa.h"

namespace jfa {

constexpr int kTile = 128;  // rows of a Q or K/V tile (tcgen05 M = 128)

// Programmatic dependent launch. The kernels of one entry point run as a chain
// on the caller's stream (status clear, queue, pre-pass, main kernel,
// post-pass); each later kernel is launched so that it may be scheduled while
// the one before it finishes, and it calls wait_prior_grid() before it touches
// anything that kernel wrote (the wait returns once the prior grid has
// completed and its writes are visible). A kernel calls allow_next_grid()
// once every block of it has started, which lets the next one be scheduled.
// Every kernel launched this way waits before it exits, so completion is
// ordered along the chain.
template <class... KArgs, class... Args>
inline cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
#ifdef __CUDACC__
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif

// Runs `set` (a kernel attribute call, idempotent) once per device: `done`
// holds one bit per device already set, so launches from several threads or
// on several devices stay correct. Devices past 63 run it on every launch.
template <class F>
inline cudaError_t once_per_device(std::atomic<uint64_t>& done, F&& set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? uint64_t(1) << dev : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = set();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Where a pipeline wait gave up (second word of the device status block).
enum WaitSite : int32_t {
  kSiteFwdProdQ = 101,
  kSiteFwdProdSlot = 102,
  kSiteFwdMmaQ = 111,
  kSiteFwdMmaSlot = 112,
  kSiteFwdMmaP = 113,
  kSiteFwdMmaOFree = 114,
  kSiteFwdSoftS = 121,
  kSiteFwdSoftO = 122,
  kSiteFwdSoftMl = 123,
  kSiteFwdDrain = 131,
  kSiteFwdEpi = 141,
  kSiteBwdProdKV = 201,
  kSiteBwdProdQ = 202,
  kSiteBwdMmaKV = 211,
  kSiteBwdMmaQ = 212,
  kSiteBwdMmaP = 213,
  kSiteBwdMmaDS = 214,
  kSiteBwdMmaDQFree = 215,
  kSiteBwdMmaAccFree = 216,
  kSiteBwdSoftS = 221,
  kSiteBwdSoftDP = 222,
  kSiteBwdDQ = 231,
  kSiteBwdEpi = 241,
  kSiteBwdDrain = 251,
  // checks of a debug build (JFA_ERR_BAD_INPUT): a tile outside its sequence or head
  kSiteCheckFwdQ = 161,
  kSiteCheckFwdKV = 162,
  kSiteCheckBwdKV = 261,
  kSiteCheckBwdQ = 262,
  kSiteQueueOffsets = 301,
  kSiteDecodeTable = 401,
  kSiteSelftestInput = 901,  // the self-test's first stage (its input never arrives)
  kSiteSelftestChain = 902,  // the self-test's second stage (should leave through the abort flag)
};

// Device status block at the start of every workspace (256 bytes).
//   [0] status (jfa_status), [1] detail (WaitSite or check code),
//   [2] number of queued work items.
constexpr size_t kStatusBytes = 256;
// Status word counting the work items handed out on demand (zeroed with the block).
constexpr int kStatusItemCounter = 8;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Queue modes: which tiles are work items and what each costs.
enum QueueMode : int32_t {
  kQueueSelfFwd = 0,   // items (b, h, q-tile); cost = kv tiles visited
  kQueueSelfBwd = 1,   // items (b, h, kv-tile); cost = q tiles visited
  kQueueBcastFwd = 2,  // items (b, h, q-tile of the shared Q); cost = kv tiles of b
  kQueueBcastBwd = 3,  // items (b, h, kv-tile of b); cost = q tiles of the shared Q
  // Varlen / GQA: offsets = query offsets, k_offsets = key offsets; causal is
  // bottom-right aligned. Items of cost 0 are kept (their outputs are zeros).
  kQueueVarFwd = 4,    // items (b, query head, q-tile); cost = key tiles visited
  kQueueVarBwd = 5,    // items (b, KV head, kv-tile); cost = group x q tiles visited
};

__host__ __device__ inline bool queue_var(int mode) { return mode == kQueueVarFwd || mode == kQueueVarBwd; }

struct QueueParams {
  const int32_t* offsets;  // [batch+1] (varlen: query offsets)
  const int32_t* k_offsets;  // varlen only: key offsets [batch+1]
  int32_t batch, heads, total, max_seqlen, causal, mode, q_len;
  int32_t total_k, max_seqlen_k, group;  // varlen only (group = q_heads / kv_heads)
  int32_t* status;         // status block
  int32_t* tile_base;      // [batch+1] exclusive prefix of q-tiles (self modes)
  int4* items;             // (b, h, t, cost); varlen backward: (b, h, t, query tile_base of b)
  int4* item_seq;          // optional: (first row, length, tile_base) of each item's sequence;
                           // varlen: (first query row, L_q, first key row, L_k)
  int32_t max_items;
  int32_t count_index;     // status word that receives the number of items; the next word
                           // receives the number with cost >= 1 (they come first)
};

// Work-item bound used to size the queue: sum_b ceil(L_b/128) <= ceil(total/128) + batch.
inline int64_t max_tiles(int64_t total, int64_t batch) { return (total + kTile - 1) / kTile + batch; }

struct BwdLaunch {
  int head_dim, head_chunk;
  const int32_t* offsets;
  const int32_t* tile_base;
  const int4* items;
  const int4* item_seq;  // (first row, length, tile_base) of each item's sequence
  int32_t* status;
  const float* lse2p;
  const float* deltap;
  float* dq_acc;
  void* dk;
  void* dv;
  int heads, total, bcast, q_len, causal, pad_tiles;
  int var, group, kv_heads;  // varlen: items carry query and key bounds; q_heads / kv_heads
  int col0;      // first head-dim column of this launch's slices (0 unless a pass covers part of d)
  int n_chunks;  // slices per item in this launch (0: head_dim / head_chunk)
  float scale;
  uint64_t budget_ns;
  int grid;
};

// Varlen / GQA description handed to the forward launchers (var = 0: the
// self-attention or broadcast-Q item records).
struct VarInfo {
  int var = 0;
  int group = 1;
};

// Launchers (defined in the kernel translation units).
cudaError_t launch_queue(const QueueParams& p, cudaStream_t stream);
cudaError_t launch_fwd(int head_dim, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const int32_t* offsets, const int4* items, const int4* item_seq, const VarInfo& var,
                       int32_t* status, void* o, float* lse, int heads, int total, int bcast, int q_len, float scale,
                       uint64_t budget_ns, int grid, cudaStream_t stream);
// Flat-stream forward (head_dim 128); items from the plain forward queue modes,
// K and V read in 128-row boxes, O (to) written in 64-column x 128-row boxes.
cudaError_t launch_fwd_stream(bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, const int4* items, const int4* item_seq, const VarInfo& var,
                              int32_t* status, void* o, float* lse, int heads, int total, int bcast, int q_len,
                              float scale, uint64_t budget_ns, int grid, cudaStream_t stream);
// tdq: the fp32 dQ accumulator [rows, H*D] in 32-column x 128-row boxes, 128B swizzle.
// tdk, tdv: dK and dV (bf16 [rows, H*D]) in 64-column x 128-row boxes, 128B swizzle.
cudaError_t launch_bwd_main(const BwdLaunch& L, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, cudaStream_t stream);
// Also zeroes the fp32 dQ accumulator dq_acc ([rows, H*D]: the sequences' rows, or the
// shared Q's rows for broadcast-Q).
cudaError_t launch_bwd_pre(int head_dim, const void* o, const void* dout, const float* lse, const int32_t* offsets,
                           const int32_t* tile_base, const int32_t* status, int batch, int heads, int total, int bcast,
                           int q_len, int pad_tiles, int grid_tiles, float* lse2p, float* deltap, float* dq_acc,
                           cudaStream_t stream);
cudaError_t launch_bwd_post(const float* acc, void* dq, int64_t n, float scale, const int32_t* status, int sms,
                            cudaStream_t stream);
// FP8 (e4m3) input forward, head_dim 128: V transposed per 128-key tile into
// [128 head-dim rows x 128 keys] blocks (block g * H + h = key tile g, head h;
// tiles numbered by tile_base), one CTA per item of the self-attention forward
// queue, then the forward over that queue.
// inv_descale non-null: v is bf16, quantized on the way to e4m3(v * *inv_descale).
cudaError_t launch_vt_transpose(const void* v, const int4* items, const int4* item_seq, const int32_t* status,
                                int heads, int max_items, void* vt, cudaStream_t stream,
                                const float* inv_descale = nullptr);
cudaError_t launch_fwd_fp8(bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const CUtensorMap& to, const int4* items, const int4* item_seq, int32_t* status, void* o, float* lse, int heads,
                           int total, float s_log2, float v_descale, uint64_t budget_ns, int grid,
                           cudaStream_t stream);
// Failure-detection self-test: one CTA whose first pipeline stage waits for an
// input that never arrives; status[4] = 1 when the second stage left through
// the abort flag.
cudaError_t launch_selftest_wait(int32_t* status, uint64_t budget_ns, cudaStream_t stream);
cudaError_t launch_decode(const jfa_decode_args& a, float* part_o, float* part_lse, int32_t* status,
                          cudaStream_t stream);
// The split-KV decode with q_len query tokens per sequence and optional
// per-sequence split counts (min_split_tokens > 0); launch_decode is q_len 1,
// min_split_tokens 0. Partials: part_o [S, B, q_len, Hq, 128], part_lse [S, B, q_len, Hq].
struct DecodeLaunch {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* page_table;
  const int32_t* seqlens_k;
  int32_t batch, q_len, q_heads, kv_heads, page_size, num_pages, max_pages, num_splits, min_split_tokens;
  float scale;
  void* o;
  float* lse;
  int32_t* split_bounds_out;
  int32_t* split_counts_out;
  void* main_kernel_events;
};
cudaError_t launch_decode_general(const DecodeLaunch& a, float* part_o, float* part_lse, int32_t* status,
                                  cudaStream_t stream);
// Clears a call's status block (a kernel, not a memset, so that the call's next
// kernel can start as its programmatic dependent).
cudaError_t launch_status_clear(int32_t* status, cudaStream_t stream);
#ifdef JFA_TRACE
// Registers the trace buffer that later calls' status blocks carry (nullptr: off):
// `ctas` CTA slots of 16 warp slots of `records_per_warp` records.
void set_trace_buffer(void* buffer, int32_t records_per_warp, int32_t ctas);
#endif
// Argument checks of jfa_decode_splitkv (scalars, alignment), without the workspace.
jfa_status check_decode_args(const jfa_decode_args* a);

}  // namespace jfa
