/*
 * jfa.h -- C ABI of the jagged FlashAttention library for GB300 (sm_103a).
 *
 * Exact attention over variable-length ("jagged") sequences packed back to
 * back with an int32 offsets tensor and no padding tokens, its recompute-based
 * backward, a broadcast-Q variant whose dQ is summed over the batch, a varlen
 * form with separate query / key lengths and grouped KV heads, and a split-KV
 * decode (one or a few query tokens per sequence) over a paged, grouped-query
 * KV cache.
 *
 * Sources of the operations (web pages; cited by title and section):
 *  [JFA]  "Optimizing Jagged Flash Attention with TLX: The Road Toward SOTA FA4
 *         on Blackwell" (aivexanews): jagged packing with an offsets tensor,
 *         broadcast-Q with dQ summed across the batch (third paragraph);
 *         persistent, warp-specialised CTAs (fourth paragraph); jagged tile
 *         load balancing, loop peeling, dQ reduce staging (fifth paragraph).
 *  [B300] "Cutting-edge isn't plug-and-play: customizing FA4 on B300"
 *         (TwelveLabs): FlashAttention recap (tiling is exact); Phase 1
 *         (single-buffered TMEM forward); Phase 2 (head-axis chunked backward
 *         and its pseudocode: S, dP rebuilt per tile, P from the saved LSE,
 *         "delta", dS); bug hunting (single-stage producer/consumer order).
 *  [INF]  "Optimizing FlashAttention-4 for Efficient Inference" (hpjadul):
 *         PR 1940 (parallelism across the KV dimension), PR 1999 / PR 2104
 *         (KV pages of arbitrary size), PR 2186 (GQA packing), PR 1993 (tiles
 *         sized to few query rows).
 *
 * Conventions shared by every entry point
 *  - Tensors are dense, row-major, in device memory unless stated otherwise.
 *    "bf16" is IEEE bfloat16; "[a, b, c]" lists dimensions outermost first.
 *  - Jagged tensors are [total, heads, head_dim]: sequence b owns rows
 *    offsets[b] .. offsets[b+1]-1. offsets is int32 [batch+1] on the device
 *    with offsets[0] = 0, non-decreasing, offsets[batch] = total.
 *  - LSE is the natural-log log-sum-exp of the scaled scores of each query row.
 *  - Every pointer must be 16-byte aligned (TMA and 16-byte vector access);
 *    head_dim must be 64, 128 or 192 unless stated otherwise.
 *  - Every pointer is device memory of the current device (cudaGetDevice()
 *    when the call is made), and each buffer spans at least the extent its
 *    field comment gives for the sizes in the argument struct. The library
 *    checks null pointers, alignment and the sizes themselves, but cannot see
 *    an allocation's extent: a shorter buffer is read or written out of bounds.
 *  - The caller owns and allocates every buffer, including the workspace,
 *    whose size comes from the matching *_workspace_size() call. The library
 *    allocates no memory, keeps no per-call state between calls, and may be
 *    called from several host threads on different streams with separate
 *    workspaces. Concurrent calls that share a workspace race. (Its only
 *    process-wide state is set-once: each kernel's shared-memory limit, raised
 *    once per device, and cached device properties.)
 *  - All work is enqueued on `stream`; no call synchronises the stream except
 *    jfa_read_device_status(). Host-side argument errors are returned before
 *    anything is enqueued. Problems only the device can see (malformed
 *    offsets or page table, a pipeline wait that ran out of time) are written
 *    to a status word in the workspace, read back by jfa_read_device_status().
 *  - max_seqlen / total arguments are host copies of facts about the device
 *    offsets, so that no device-to-host copy is needed; the kernels check
 *    them against the offsets and report JFA_ERR_BAD_INPUT on a mismatch.
 *  - A call enqueues a short chain of kernels (a status clear, the work
 *    queue, the pass's kernels). Every kernel after the first is launched with
 *    programmatic stream serialization: it may be scheduled while the one
 *    before it finishes and waits for it on the device before reading its
 *    results, so the chain keeps stream order and can be captured in a graph.
 *  - main_kernel_events: optional pair of cudaEvent_t (may be NULL). When
 *    set, event [0] is recorded on `stream` just before the main attention
 *    kernel and event [1] just after it, so a caller can time that kernel
 *    alone (the recorded events keep the main kernel from starting before
 *    the kernel in front of it has finished). The library does not create,
 *    own or destroy them.
 */
#ifndef JFA_H
#define JFA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define JFA_API __attribute__((visibility("default")))
#else
#define JFA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  JFA_OK = 0,
  JFA_ERR_INVALID_ARG = 1,          /* null/misaligned pointer, bad size, ... */
  JFA_ERR_UNSUPPORTED = 2,          /* valid request this build does not implement */
  JFA_ERR_WORKSPACE_TOO_SMALL = 3,
  JFA_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed */
  JFA_ERR_TIMEOUT = 5,              /* a device pipeline wait exceeded its time budget */
  JFA_ERR_BAD_INPUT = 6             /* device data inconsistent (offsets, page table) */
} jfa_status;

/* ------------------------------------------------------------------ forward
 * Jagged self-attention forward ([JFA] third paragraph; [B300] FlashAttention
 * recap). For every sequence b and head h:
 *   S = scale * Q_b K_b^T (causal: S_ij = -inf for j > i), P = softmax_rows(S),
 *   O_b = P V_b, LSE_i = ln sum_j exp(S_ij).
 */
typedef struct {
  const void* q;             /* bf16 [total, heads, head_dim] */
  const void* k;             /* bf16 [total, heads, head_dim] */
  const void* v;             /* bf16 [total, heads, head_dim] */
  const int32_t* offsets;    /* int32 [batch+1], device */
  int32_t batch;             /* >= 0 */
  int32_t heads;             /* >= 1 */
  int32_t head_dim;          /* 64, 128 or 192 */
  int32_t max_seqlen;        /* host: >= every L_b */
  int32_t total;             /* host: offsets[batch] */
  float scale;               /* softmax scale, e.g. 1/sqrt(head_dim) */
  int32_t causal;            /* 0 or 1 (key j visible to query i iff j <= i) */
  void* o;                   /* out: bf16 [total, heads, head_dim] */
  float* lse;                /* out: fp32 [heads, total] */
  void* main_kernel_events;  /* optional cudaEvent_t[2], see above */
} jfa_fwd_args;

/* ------------------------------------------------------------------ backward
 * Recompute-based backward ([B300] Phase 2 and its pseudocode): per tile S and
 * dP are rebuilt from Q, K, V, dO; P from S and the saved LSE; then
 *   D = rowsum(dO * O) ("delta"), dS = P * (dP - D),
 *   dV = P^T dO, dQ = scale dS K, dK = scale dS^T Q.
 * head_dim 192 runs head-axis chunked ([B300] Phase 2): each pass owns a
 * slice of dQ/dK/dV while S and dP are still accumulated over the whole head
 * dimension. By default (head_chunk 0) the slices are columns 0-127 and
 * 128-191 (two passes: TMEM holds dV and dK slices of at most 128 columns next
 * to S and dP); head_chunk 64 runs three 64-column passes.
 */
typedef struct {
  const void* q;             /* bf16 [total, heads, head_dim] */
  const void* k;             /* bf16 [total, heads, head_dim] */
  const void* v;             /* bf16 [total, heads, head_dim] */
  const void* o;             /* bf16 [total, heads, head_dim], forward output */
  const void* dout;          /* bf16 [total, heads, head_dim], gradient of O */
  const float* lse;          /* fp32 [heads, total], forward LSE */
  const int32_t* offsets;    /* int32 [batch+1], device */
  int32_t batch, heads, head_dim, max_seqlen, total;
  float scale;
  int32_t causal;
  int32_t head_chunk;        /* 0 = automatic (head_dim 192: slices of 128 and 64; else head_dim), or 64 */
  void* dq;                  /* out: bf16 [total, heads, head_dim] */
  void* dk;                  /* out: bf16 [total, heads, head_dim] */
  void* dv;                  /* out: bf16 [total, heads, head_dim] */
  void* main_kernel_events;  /* optional cudaEvent_t[2] */
} jfa_bwd_args;

/* ------------------------------------------------------------------ broadcast-Q
 * One dense Q [q_len, heads, head_dim] is the query of every sequence of a
 * jagged K/V batch ([JFA] third paragraph). Not causal.
 *   O[b] = softmax(scale Q K_b^T) V_b; backward: dQ = sum_b dQ_b (the
 *   contended cross-CTA reduction), dK_b, dV_b per sequence. The backward at
 *   head_dim 192 runs the two head-axis passes of jfa_bwd.
 */
typedef struct {
  const void* q;             /* bf16 [q_len, heads, head_dim] */
  const void* k;             /* bf16 [total_k, heads, head_dim] */
  const void* v;             /* bf16 [total_k, heads, head_dim] */
  const int32_t* kv_offsets; /* int32 [batch+1], device */
  int32_t batch, q_len, heads, head_dim, max_seqlen_k, total_k;
  float scale;
  void* o;                   /* out: bf16 [batch, q_len, heads, head_dim] */
  float* lse;                /* out: fp32 [batch, heads, q_len] */
  void* main_kernel_events;
} jfa_bcast_fwd_args;

typedef struct {
  const void* q;             /* bf16 [q_len, heads, head_dim] */
  const void* k;             /* bf16 [total_k, heads, head_dim] */
  const void* v;             /* bf16 [total_k, heads, head_dim] */
  const void* o;             /* bf16 [batch, q_len, heads, head_dim] */
  const void* dout;          /* bf16 [batch, q_len, heads, head_dim] */
  const float* lse;          /* fp32 [batch, heads, q_len] */
  const int32_t* kv_offsets;
  int32_t batch, q_len, heads, head_dim, max_seqlen_k, total_k;
  float scale;
  void* dq;                  /* out: bf16 [q_len, heads, head_dim], summed over the batch */
  void* dk;                  /* out: bf16 [total_k, heads, head_dim] */
  void* dv;                  /* out: bf16 [total_k, heads, head_dim] */
  void* main_kernel_events;
} jfa_bcast_bwd_args;

/* ------------------------------------------------------------------ varlen / GQA
 * Jagged attention whose query and key sequences have their own lengths and
 * whose query heads share KV heads ([B300] section on why the development
 * succeeded, second factor: MHA / GQA / MQA head layouts, causal and
 * non-causal masks and varlen packing are the surface the kernel must cover;
 * [INF] PR 2186: several query heads are processed against one KV head).
 * Sequence b has query rows q_offsets[b] .. q_offsets[b+1]-1 and key/value
 * rows k_offsets[b] .. k_offsets[b+1]-1 (L_q and L_k, either may be 0).
 * Query head h reads KV head h / (q_heads / kv_heads). For every b and h:
 *   S = scale * Q_b,h K_b,g^T, P = softmax_rows(S), O = P V_b,g,
 *   LSE_i = ln sum_j exp(S_ij).
 * causal = 1 aligns the mask to the bottom right (the pages state no
 * alignment for L_q != L_k; this is the reading where a query block is the
 * end of its key sequence): key j is visible to query i iff
 * j <= i + (L_k - L_q). With L_q == L_k this is the self-attention mask.
 * A query row that sees no key (L_k = 0, or i < L_q - L_k when causal) gets
 * O = 0 and LSE = -inf, and contributes no gradient.
 * head_dim 64, 128 or 192; q_heads must be a multiple of kv_heads. */
typedef struct {
  const void* q;              /* bf16 [total_q, q_heads, head_dim] */
  const void* k;              /* bf16 [total_k, kv_heads, head_dim] */
  const void* v;              /* bf16 [total_k, kv_heads, head_dim] */
  const int32_t* q_offsets;   /* int32 [batch+1], device */
  const int32_t* k_offsets;   /* int32 [batch+1], device */
  int32_t batch;              /* >= 0 */
  int32_t q_heads;            /* >= 1 */
  int32_t kv_heads;           /* >= 1, divides q_heads */
  int32_t head_dim;           /* 64, 128 or 192 */
  int32_t max_seqlen_q;       /* host: >= every L_q */
  int32_t max_seqlen_k;       /* host: >= every L_k */
  int32_t total_q;            /* host: q_offsets[batch] */
  int32_t total_k;            /* host: k_offsets[batch] */
  float scale;
  int32_t causal;             /* 0, or 1 = bottom-right aligned (see above) */
  void* o;                    /* out: bf16 [total_q, q_heads, head_dim] */
  float* lse;                 /* out: fp32 [q_heads, total_q] */
  void* main_kernel_events;   /* optional cudaEvent_t[2] */
} jfa_varlen_fwd_args;

/* Backward of jfa_fwd_varlen (same recompute scheme as jfa_bwd). dK and dV of
 * a KV head are summed over the q_heads / kv_heads query heads that read it
 * (accumulated on chip, no atomics); dQ as in jfa_bwd. head_dim 192 runs
 * head-axis chunked as in jfa_bwd. */
typedef struct {
  const void* q;              /* bf16 [total_q, q_heads, head_dim] */
  const void* k;              /* bf16 [total_k, kv_heads, head_dim] */
  const void* v;              /* bf16 [total_k, kv_heads, head_dim] */
  const void* o;              /* bf16 [total_q, q_heads, head_dim], forward output */
  const void* dout;           /* bf16 [total_q, q_heads, head_dim] */
  const float* lse;           /* fp32 [q_heads, total_q], forward LSE */
  const int32_t* q_offsets;   /* int32 [batch+1], device */
  const int32_t* k_offsets;   /* int32 [batch+1], device */
  int32_t batch, q_heads, kv_heads, head_dim;
  int32_t max_seqlen_q, max_seqlen_k, total_q, total_k;
  float scale;
  int32_t causal;
  int32_t head_chunk;         /* 0 = automatic (as in jfa_bwd_args), or 64 */
  void* dq;                   /* out: bf16 [total_q, q_heads, head_dim] */
  void* dk;                   /* out: bf16 [total_k, kv_heads, head_dim] */
  void* dv;                   /* out: bf16 [total_k, kv_heads, head_dim] */
  void* main_kernel_events;   /* optional cudaEvent_t[2] */
} jfa_varlen_bwd_args;

/* ------------------------------------------------------------------ paged decode
 * One query token per sequence against a paged KV cache ([INF] PR 1999/2104:
 * pages of any size >= 1; PR 2186: the q_heads/kv_heads query heads that share
 * a KV head are processed together; PR 1940: the KV range of each sequence is
 * split into num_splits parts processed in parallel, then merged).
 * Token t of sequence b lives in page page_table[b][t / page_size], slot
 * t % page_size; query head h reads KV head h / (q_heads / kv_heads).
 * Split s of sequence b covers tokens [s*c, min((s+1)*c, L_b)) with
 * c = ceil(L_b / num_splits). The merge is
 *   lse = ln sum_s exp(lse_s), O = sum_s exp(lse_s - lse) O_s.
 * A sequence with L_b = 0 gets O = 0 and LSE = -inf.
 * head_dim must be 128; q_heads / kv_heads must be 1, 2, 4, 8 or 16.
 */
typedef struct {
  const void* q;             /* bf16 [batch, q_heads, head_dim] */
  const void* k_cache;       /* bf16 [num_pages, page_size, kv_heads, head_dim] */
  const void* v_cache;       /* bf16 [num_pages, page_size, kv_heads, head_dim] */
  const int32_t* page_table; /* int32 [batch, max_pages]; entries past ceil(L_b/page_size) are not read */
  const int32_t* seqlens_k;  /* int32 [batch], 0 <= L_b <= max_pages*page_size */
  int32_t batch, q_heads, kv_heads, head_dim;
  int32_t page_size;         /* >= 1 */
  int32_t num_pages;         /* page_table entries must be < num_pages */
  int32_t max_pages;
  int32_t num_splits;        /* 1 .. 128 */
  float scale;
  void* o;                   /* out: bf16 [batch, q_heads, head_dim] */
  float* lse;                /* out: fp32 [batch, q_heads] */
  int32_t* split_bounds_out; /* optional out: int32 [batch, num_splits, 2] (start, end) */
  void* main_kernel_events;  /* optional cudaEvent_t[2] around the split kernel */
} jfa_decode_args;

/* ------------------------------------------------------------------ FP8 forward
 * Jagged self-attention forward with FP8 inputs ([INF] PR 2109: FP8 inputs for
 * inference). The page gives no format or scale convention; reading: e4m3
 * bytes (sign, 4 exponent bits with bias 7, 3 mantissa bits) with one descale
 * factor per tensor, so byte x of Q stands for e4m3(x) * q_descale (likewise
 * K, V), and the forward computes jfa_fwd's attention over those values:
 *   S = scale * Q_b K_b^T (causal: j <= i), P = softmax_rows(S), O = P V_b.
 * P enters P V as e4m3 (relative rounding error up to 2^-4); O is bf16, LSE
 * fp32 natural log. head_dim must be 128. */
typedef struct {
  const void* q;             /* e4m3 bytes [total, heads, 128] */
  const void* k;             /* e4m3 bytes [total, heads, 128] */
  const void* v;             /* e4m3 bytes [total, heads, 128] */
  const int32_t* offsets;    /* int32 [batch+1], device */
  int32_t batch, heads, head_dim, max_seqlen, total;
  float scale;
  int32_t causal;
  float q_descale, k_descale, v_descale;  /* > 0 */
  void* o;                   /* out: bf16 [total, heads, 128] */
  float* lse;                /* out: fp32 [heads, total] */
  void* main_kernel_events;  /* optional cudaEvent_t[2] */
  const void* vt;            /* optional: V already in the forward's key-contiguous layout, as
                                jfa_fp8_quantize_v writes it for the same offsets and heads (v is
                                then not read and may be NULL, and the call makes no pass over V) */
} jfa_fwd_fp8_args;

/* V for the FP8 forward, quantized straight into the layout the forward reads
 * ([INF] PR 2109; the layout is this library's). P V takes V as a K-major
 * operand (keys contiguous), so jfa_fwd_fp8 rewrites an e4m3 [total, heads,
 * 128] V on every call as one [128 dims x 128 keys] block per 128-key tile of
 * each sequence and head. A caller that quantizes V from bf16 anyway can write
 * those blocks instead: this call reads bf16 V and writes
 *   block (tile_base[b] + t) * heads + h, byte [d][k] = e4m3(V[s_b + 128 t + k, h, d] * inv)
 * with inv = 1 / v_descale rounded to fp32, e4m3 rounding to nearest even and
 * saturating at +-448, tile_base[b] = sum over b' < b of ceil(L_b' / 128), and
 * zero bytes for keys past the end of the sequence; jfa_fwd_fp8 with vt set
 * (and the same v_descale) then reads them. vt must hold
 * jfa_fp8_vt_bytes(batch, heads, total) bytes (16-byte aligned); head_dim must
 * be 128. */
typedef struct {
  const void* v;             /* bf16 [total, heads, 128] */
  const int32_t* offsets;    /* int32 [batch+1], device */
  int32_t batch, heads, head_dim, max_seqlen, total;
  float v_descale;           /* > 0 */
  void* vt;                  /* out: e4m3 blocks */
} jfa_fp8_quantize_v_args;

/* ------------------------------------------------------------------ small-query paged decode
 * Paged split-KV GQA decode with q_len >= 1 query tokens per sequence ([INF]
 * PR 1993: tiles sized to few query rows, e.g. speculative decoding; with the
 * paging, KV splitting and GQA packing of jfa_decode_splitkv). Reading (the
 * page gives no layout): the q_len new tokens of sequence b are the last q_len
 * tokens of its cache (L_b already counts them); query token i sits at key
 * position L_b - q_len + i and sees keys j <= L_b - q_len + i. A query row
 * that sees no key (L_b < q_len - i) gets O = 0, LSE = -inf.
 * The q_len x (q_heads / kv_heads) (token, head) rows of one KV head form one
 * tile; that product must be <= 16.
 * Splits: with min_split_tokens = 0 every sequence takes num_splits parts;
 * with min_split_tokens > 0 sequence b takes
 *   S_b = clamp(ceil(L_b / min_split_tokens), 1, num_splits)
 * parts (short sequences are not spread thin); part s < S_b covers
 * [s c_b, min((s+1) c_b, L_b)) with c_b = ceil(L_b / S_b), parts s >= S_b are
 * empty, reported as (L_b, L_b). The merge is that of jfa_decode_splitkv.
 * head_dim must be 128. */
typedef struct {
  const void* q;              /* bf16 [batch, q_len, q_heads, head_dim] */
  const void* k_cache;        /* bf16 [num_pages, page_size, kv_heads, head_dim] */
  const void* v_cache;        /* bf16 [num_pages, page_size, kv_heads, head_dim] */
  const int32_t* page_table;  /* int32 [batch, max_pages] */
  const int32_t* seqlens_k;   /* int32 [batch], 0 <= L_b <= max_pages*page_size, new tokens included */
  int32_t batch, q_len, q_heads, kv_heads, head_dim;
  int32_t page_size, num_pages, max_pages;
  int32_t num_splits;         /* 1 .. 128: split slots (the upper bound of S_b) */
  int32_t min_split_tokens;   /* 0, or the fewest tokens per part when choosing S_b */
  float scale;
  void* o;                    /* out: bf16 [batch, q_len, q_heads, head_dim] */
  float* lse;                 /* out: fp32 [batch, q_len, q_heads] */
  int32_t* split_bounds_out;  /* optional out: int32 [batch, num_splits, 2] */
  int32_t* split_counts_out;  /* optional out: int32 [batch], S_b */
  void* main_kernel_events;   /* optional cudaEvent_t[2] around the split kernel */
} jfa_decode_smallq_args;

/* Workspace sizes in bytes (0 only when args is NULL). */
JFA_API size_t jfa_fwd_workspace_size(const jfa_fwd_args* args);
JFA_API size_t jfa_bwd_workspace_size(const jfa_bwd_args* args);
JFA_API size_t jfa_bcast_fwd_workspace_size(const jfa_bcast_fwd_args* args);
JFA_API size_t jfa_bcast_bwd_workspace_size(const jfa_bcast_bwd_args* args);
JFA_API size_t jfa_decode_workspace_size(const jfa_decode_args* args);
JFA_API size_t jfa_varlen_fwd_workspace_size(const jfa_varlen_fwd_args* args);
JFA_API size_t jfa_varlen_bwd_workspace_size(const jfa_varlen_bwd_args* args);
JFA_API size_t jfa_decode_smallq_workspace_size(const jfa_decode_smallq_args* args);
JFA_API size_t jfa_fwd_fp8_workspace_size(const jfa_fwd_fp8_args* args);
JFA_API size_t jfa_fp8_quantize_v_workspace_size(const jfa_fp8_quantize_v_args* args);
/* Bytes of the V blocks for a batch (an upper bound: (ceil(total/128) + batch) x heads x 16384). */
JFA_API size_t jfa_fp8_vt_bytes(int32_t batch, int32_t heads, int32_t total);

/* Entry points. `workspace` is device memory of at least the size above,
 * 256-byte aligned; its contents on entry do not matter. */
JFA_API jfa_status jfa_fwd(const jfa_fwd_args* args, void* workspace, size_t workspace_bytes, cudaStream_t stream);
JFA_API jfa_status jfa_bwd(const jfa_bwd_args* args, void* workspace, size_t workspace_bytes, cudaStream_t stream);
JFA_API jfa_status jfa_fwd_broadcast_q(const jfa_bcast_fwd_args* args, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);
JFA_API jfa_status jfa_bwd_broadcast_q(const jfa_bcast_bwd_args* args, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);
JFA_API jfa_status jfa_decode_splitkv(const jfa_decode_args* args, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);
JFA_API jfa_status jfa_fwd_varlen(const jfa_varlen_fwd_args* args, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);
JFA_API jfa_status jfa_bwd_varlen(const jfa_varlen_bwd_args* args, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);
JFA_API jfa_status jfa_decode_smallq(const jfa_decode_smallq_args* args, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream);
JFA_API jfa_status jfa_fwd_fp8(const jfa_fwd_fp8_args* args, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);
JFA_API jfa_status jfa_fp8_quantize_v(const jfa_fp8_quantize_v_args* args, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

/* Paged split-KV decode that allocates nothing. The pages have no
 * counterpart for this entry point; it exists for callers that cannot
 * allocate device memory at call time (a plugin handed only its input and
 * output buffers by a host runtime, or a serving path whose memory is planned
 * up front and must not allocate or free). Same arguments and results as
 * jfa_decode_splitkv, but the split partials live in a fixed scratch array
 * inside the library (about 16.1 MiB per GPU, held until the process exits):
 *  - num_splits * batch * q_heads must be <= 32768, else the call returns
 *    JFA_ERR_WORKSPACE_TOO_SMALL before enqueueing anything;
 *  - the first call on a device looks up the scratch address for that device
 *    (make that first call before any stream capture on the device);
 *  - calls no cudaMalloc / cudaFree and no allocating library routine;
 *  - every call shares the scratch: calls whose work overlaps on the GPU race,
 *    so serialise them (one stream, or explicit ordering);
 *  - the scratch address is looked up once per CUDA context (a context
 *    recreated after cudaDeviceReset, or a second context on the device, gets
 *    its own lookup);
 *  - arguments are checked as in jfa_decode_splitkv before the size limit, so
 *    a malformed request returns JFA_ERR_INVALID_ARG / JFA_ERR_UNSUPPORTED;
 *  - device-detected input errors (a page entry out of range) are handled in
 *    the kernel as in jfa_decode_splitkv and recorded in the status word of
 *    the internal scratch: read them with jfa_decode_noalloc_status. */
JFA_API jfa_status jfa_decode_splitkv_noalloc(const jfa_decode_args* args, cudaStream_t stream);

/* Device status of the last jfa_decode_splitkv_noalloc call on the current
 * context, as jfa_read_device_status returns it for a workspace: synchronises
 * `stream`, then returns JFA_OK, JFA_ERR_TIMEOUT or JFA_ERR_BAD_INPUT (with a
 * check code in *detail, optional), or JFA_ERR_CUDA. Allocates nothing. No
 * counterpart on the pages either. */
JFA_API jfa_status jfa_decode_noalloc_status(cudaStream_t stream, int32_t* detail);

/* Failure-detection self-test ([B300] bug hunting: a producer/consumer
 * pipeline that deadlocked). Every pipeline wait in this library is bounded in
 * time; when one runs out, the kernel records JFA_ERR_TIMEOUT and the waiting
 * site in the workspace status word, raises its CTA's abort flag so that every
 * other role leaves as well, and returns, leaving the CUDA context usable.
 * This entry point runs that path on purpose: a one-CTA kernel whose first
 * stage waits budget_us microseconds (1 .. 10^7) for an input that never
 * arrives, while its second stage waits for the first with an 8x longer
 * budget. Afterwards jfa_read_device_status(workspace) returns
 * JFA_ERR_TIMEOUT with detail 901 (the first stage's wait), and the 32-bit
 * word at byte offset 16 of the workspace is 1 when the second stage left
 * through the abort flag before its own budget. workspace: >= 256 bytes of
 * device memory, 256-byte aligned. */
JFA_API jfa_status jfa_selftest_wait_timeout(int32_t budget_us, void* workspace, cudaStream_t stream);

/* Synchronises `stream`, then returns the device status word of the last call
 * that used `workspace` (JFA_OK, JFA_ERR_TIMEOUT or JFA_ERR_BAD_INPUT), or
 * JFA_ERR_CUDA if the stream reports an error. *detail (optional) receives a
 * code naming the wait or check that failed. */
JFA_API jfa_status jfa_read_device_status(const void* workspace, cudaStream_t stream, int32_t* detail);

/* Per-role event trace of the persistent kernels (the head_dim 128 forward
 * of jfa_fwd / jfa_fwd_broadcast_q / jfa_fwd_varlen and every backward), for
 * looking into the warp-specialised pipelines ("Cutting-edge isn't
 * plug-and-play: customizing FA4 on B300", bug hunting: a producer/consumer
 * deadlock). Only a library built with JFA_TRACE records; jfa_trace_compiled()
 * returns 1 there and 0 otherwise, where jfa_trace_enable returns
 * JFA_ERR_UNSUPPORTED and the kernels hold no trace code.
 *  - buffer: device memory, 16-byte aligned, owned by the caller, of at least
 *    SMs x 16 x records_per_warp x 32 bytes (SMs of the current device; else
 *    JFA_ERR_INVALID_ARG); zero it before each call to be recorded.
 *  - Layout: [CTA][warp slot 0..15][records_per_warp] records of 32 bytes:
 *    uint64 clock64 (SM cycles), uint64 globaltimer (ns), uint32 event
 *    (kernel << 16 | code: kernel 1 = forward, 2 = backward; the codes are
 *    listed in varlen_flashattention_gb300/trace.py), uint32 argument (step or
 *    item counter of the CTA), uint32 SM id, uint32 0. A warp's records are in
 *    program order; the first all-zero record ends them; records past
 *    records_per_warp are dropped.
 *  - Each traced kernel launch writes from the start of every slot, so the
 *    buffer holds the last one (for head_dim 192, the second head-axis pass).
 *  - The setting is process-wide and applies to calls enqueued after it;
 *    jfa_trace_enable(NULL, 0, 0) turns recording off. */
JFA_API jfa_status jfa_trace_enable(void* buffer, size_t bytes, int32_t records_per_warp);
JFA_API int32_t jfa_trace_compiled(void);

/* Static string for a status code. */
JFA_API const char* jfa_status_string(jfa_status status);

/* Library version, as major*10000 + minor*100 + patch. */
JFA_API int32_t jfa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* JFA_H */
