// Split-KV paged GQA decode: one or a few query tokens per sequence against a
// KV cache addressed through a page table, the KV range split into parallel
// parts whose partial softmax results are merged by a second kernel.
//
// Sources: "Optimizing FlashAttention-4 for Efficient Inference" (hpjadul),
// sections PR 1940 (parallelism across the KV dimension), PR 1999 / PR 2104
// (KV pages of any size), PR 2186 (GQA packing: the query heads that share a
// KV head are processed in one tile so K/V are read once) and "Key
// Enhancements" (irregular gathers use per-thread asynchronous loads rather
// than bulk tensor copies).
//
// Design (GB300): the path is bound by HBM reads of K and V (about 0.5 flop
// per byte), so the kernel is organised around memory-level parallelism:
// every lane copies its 16-byte pieces of whole 256-byte cache rows with
// cp.async into a private slot of a per-warp ring of kDecStages 16-token
// blocks, so each warp keeps kDecStages - 1 blocks in flight while it
// computes one; the GQA group of query heads rides along as the rows of an
// m16n8k16 register MMA. The MMA is used to cut issue slots (no shuffle
// reductions), not for its FLOPs; tcgen05's 64/128-row tiles would waste more
// of the tensor core on 1..16 real rows than this does. A lane only reads
// back the pieces it copied, so the ring needs no synchronisation beyond the
// lane's own cp.async groups, and its layout (piece j of lane l at
// [j][l]) makes every warp-wide copy and read 512 contiguous bytes.
//
// Several query tokens ("Optimizing FlashAttention-4 for Efficient
// Inference", PR 1993: tiles sized to few query rows): the q_len new tokens of
// a sequence are its last q_len cache positions; query i sits at key position
// L - q_len + i and sees keys up to it. The rows of the MMA tile are the
// (token, head) pairs of one KV head, row r = token (r / G), head (r % G), at
// most 16 rows; each row carries its own causal limit. A split count may be
// chosen per sequence: S_b = clamp(ceil(L_b / min_split_tokens), 1, S).
//
// Index mappings used below (each lane: g = lane / 4, q = lane % 4):
//  * QK^T: head dimension permuted so that each lane's four k-values of
//    k-steps 2c' and 2c'+1 are the 8 contiguous bf16 at d = 32c' + 8q;
//    Q is loaded with the same permutation, so dot products are unchanged.
//  * PV: output column n = g of n-tile j is head-dimension d = 16g + j, so a
//    lane reads 32 contiguous bytes of each V row it needs; the permutation
//    is undone when the partial result is written.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "jfa_internal.h"
#include "ptx.cuh"

namespace jfa {

struct DecodeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  const int32_t* page_table;
  const int32_t* seqlens;
  int32_t batch, hq, hkv, page_size, num_pages, max_pages, num_splits;
  int32_t q_len;        // query tokens per sequence (rows of a tile: G * q_len <= 16)
  int32_t min_split;    // > 0: per-sequence split count clamp(ceil(L / min_split), 1, num_splits)
  int32_t* counts_out;  // optional [B]: the split count of each sequence
  float scale_log2;
  float* part_o;        // [S, B, q_len, Hq, 128], normalised within the split
  float* part_lse;      // [S, B, q_len, Hq], natural log, -inf when empty
  int32_t* bounds_out;  // optional [B, S, 2]
  int32_t* status;
};

constexpr int kDecD = 128;
constexpr int kDecWarps = 4;
// Blocks per warp ring: two (one in flight while one is computed) at three
// CTAs per SM measured faster than three at two CTAs per SM (4.61 against
// 4.43 TB/s at page 16, 16 splits): more CTAs per SM overlap one CTA's start
// and final merge with the others' loops, which deeper rings did not make up.
constexpr int kDecStages = 2;
constexpr int kDecRingBytes = kDecStages * kDecWarps * 16 * 32 * 16;  // 16 pieces x 32 lanes x 16 B

// 16-byte asynchronous global -> shared copy; bytes past src_bytes are zero.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(ptx::smem_u32(smem_dst)), "l"(gsrc),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void flag_bad(int32_t* status, int32_t code) {
  if (atomicCAS(status, JFA_OK, JFA_ERR_BAD_INPUT) == JFA_OK) status[1] = code;
}

constexpr int kDecMaxSplits = 128;  // the entry points accept at most 128 splits

// Merge of the S split partials of one output row (one warp):
// lse = ln sum_s exp(lse_s), O = sum_s exp(lse_s - lse) O_s. The split
// weights go through shared memory (0 for an empty split, whose partial O is
// zero); each lane sums four output columns over the splits in order, with
// the loads of sixteen splits in flight at a time. Partials are read with
// L2-only loads (other SMs wrote them).
__device__ __forceinline__ void merge_row(const float* part_o, const float* part_lse, int S, int64_t stride,
                                          int64_t row, int lane, float* s_w, __nv_bfloat16* o, float* lse) {
  constexpr float kLog2e = 1.4426950408889634f;
  float ls[kDecMaxSplits / 32];
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kDecMaxSplits / 32; ++k) {
    const int s = lane + 32 * k;
    ls[k] = s < S ? __ldcg(part_lse + s * stride + row) : -INFINITY;
    M = fmaxf(M, ls[k]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
#pragma unroll
  for (int k = 0; k < kDecMaxSplits / 32; ++k) {
    const int s = lane + 32 * k;
    if (s < S) s_w[s] = (M == -INFINITY || ls[k] == -INFINITY) ? 0.f : ptx::ex2((ls[k] - M) * kLog2e);
  }
  __syncwarp();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float Z = 0.f;
  for (int s0 = 0; s0 < S; s0 += 16) {
    float4 v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      v[j] = s0 + j < S ? __ldcg(reinterpret_cast<const float4*>(part_o + ((s0 + j) * stride + row) * kDecD) + lane)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (s0 + j >= S) break;
      const float w = s_w[s0 + j];
      Z += w;
      acc.x += w * v[j].x;
      acc.y += w * v[j].y;
      acc.z += w * v[j].z;
      acc.w += w * v[j].w;
    }
  }
  __syncwarp();  // s_w is rewritten for the warp's next row
  const float inv = Z > 0.f ? 1.f / Z : 0.f;
  __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 c = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&a);
  packed.y = *reinterpret_cast<uint32_t*>(&c);
  *reinterpret_cast<uint2*>(o + row * kDecD + 4 * lane) = packed;
  if (lane == 0) lse[row] = Z > 0.f ? M + logf(Z) : -INFINITY;
}

// Launched as a programmatic dependent of the split kernel: its blocks may be
// scheduled while the split kernel's last blocks run, and wait here until that
// grid has completed and its partials are visible.
__global__ void __launch_bounds__(128) decode_merge_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_lse, int S, int rows,
                                                           __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  __shared__ float s_w[4][kDecMaxSplits];
  wait_prior_grid();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;  // (b, token, head)
  if (row >= rows) return;
  merge_row(part_o, part_lse, S, rows, row, lane, s_w[warp], o, lse);
}

// Rows of a tile: G query heads x q_len tokens. TWO: rows 8..15 are in use.
template <int G, bool TWO>
__global__ void __launch_bounds__(128, 3) decode_split_kernel(const DecodeParams p) {
  static_assert(G == 1 || G == 2 || G == 4 || G == 8 || G == 16, "GQA group");
  static_assert(G < 16 || TWO, "a group of 16 fills both row halves");
  constexpr bool kTwoRowHalves = TWO;
  constexpr int kRows = TWO ? 16 : 8;

  // the block ring during the loop; afterwards the per-warp partials
  extern __shared__ __align__(16) uint4 ring[];
  float(*s_o)[kRows][kDecD] = reinterpret_cast<float(*)[kRows][kDecD]>(ring);
  float(*s_m)[kRows] = reinterpret_cast<float(*)[kRows]>(reinterpret_cast<float*>(ring) + kDecWarps * kRows * kDecD);
  float(*s_l)[kRows] =
      reinterpret_cast<float(*)[kRows]>(reinterpret_cast<float*>(ring) + kDecWarps * kRows * (kDecD + 1));

  // the status block is cleared by the kernel before this one (launched as its dependent)
  wait_prior_grid();
  allow_next_grid();  // every block has started: the merge kernel may be scheduled (it waits for this grid)
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, qq = lane & 3;
  const int S = p.num_splits, P = p.page_size;
  const int QL = p.q_len, nrows = G * QL;

  int L = p.seqlens[b];
  const int64_t cap = static_cast<int64_t>(p.max_pages) * P;
  if (L < 0 || L > cap) {
    if (threadIdx.x == 0) flag_bad(p.status, kSiteDecodeTable);
    L = 0;
  }
  // this sequence's split count, then split s = [s c, min((s+1) c, L)); splits past it are empty
  int Sb = S;
  if (p.min_split > 0) Sb = max(1, min(S, static_cast<int>((static_cast<int64_t>(L) + p.min_split - 1) / p.min_split)));
  const int64_t c = (static_cast<int64_t>(L) + Sb - 1) / Sb;
  const int lo = s < Sb ? static_cast<int>(min(static_cast<int64_t>(s) * c, static_cast<int64_t>(L))) : L;
  const int hi = s < Sb ? static_cast<int>(min(static_cast<int64_t>(s + 1) * c, static_cast<int64_t>(L))) : L;
  if (p.bounds_out && kvh == 0 && threadIdx.x == 0) {
    p.bounds_out[(static_cast<int64_t>(b) * S + s) * 2 + 0] = lo;
    p.bounds_out[(static_cast<int64_t>(b) * S + s) * 2 + 1] = hi;
  }
  if (p.counts_out && s == 0 && kvh == 0 && threadIdx.x == 0) p.counts_out[b] = Sb;
  // causal limits (exclusive) of this lane's rows gq and gq + 8: token r / G sees keys < L - q_len + r / G + 1
  const int lim0 = min(hi, L - QL + gq / G + 1);
  const int lim1 = min(hi, L - QL + (gq + 8) / G + 1);

  // Q fragments (A operand, rows = (token, head) pairs of this KV group).
  uint32_t qa[8][4];
  {
    auto qrow = [&](int r) {  // row r: token r / G, head kvh * G + r % G
      return p.q + ((static_cast<int64_t>(b) * QL + r / G) * p.hq + static_cast<int64_t>(kvh) * G + r % G) * kDecD;
    };
#pragma unroll
    for (int cs = 0; cs < 8; ++cs) {
      const int d0 = 32 * (cs >> 1) + 8 * qq + 4 * (cs & 1);
      uint32_t r0a = 0, r0b = 0, r1a = 0, r1b = 0;
      if (gq < nrows) {
        const uint2 v = *reinterpret_cast<const uint2*>(qrow(gq) + d0);
        r0a = v.x;
        r0b = v.y;
      }
      if (kTwoRowHalves && gq + 8 < nrows) {
        const uint2 v = *reinterpret_cast<const uint2*>(qrow(gq + 8) + d0);
        r1a = v.x;
        r1b = v.y;
      }
      qa[cs][0] = r0a;
      qa[cs][1] = r1a;
      qa[cs][2] = r0b;
      qa[cs][3] = r1b;
    }
  }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  const int64_t row_stride = static_cast<int64_t>(p.hkv) * kDecD;  // elements between tokens of a page
  const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.max_pages;
  const int nblk = (hi - lo + 15) >> 4;

  // Copies of block kb (this warp's blocks: warp, warp + 4, ...) into ring slot `slot`:
  // pieces 0..7 = K rows g and g+8 (B operand of QK^T), 8..15 = V rows 2q, 2q+1,
  // 2q+8, 2q+9 (B operand of PV). Tokens past the split end are zero-filled
  // from an in-bounds row.
  uint4* my_ring = ring + static_cast<size_t>(warp) * kDecStages * 16 * 32;
  // Page-table entry of token lo + 16 kb + (lane % 16), read one block ahead
  // of its copies so that its latency is not in front of every block.
  auto page_entry = [&](int kb) -> int {
    const int tok = lo + kb * 16 + (lane & 15);
    return (kb < nblk && tok < hi) ? pt[tok / P] : 0;
  };
  auto issue = [&](int kb, int slot, int pg) {
    uint4* dst = my_ring + slot * 16 * 32 + lane;
    if (kb < nblk) {
      const int t0 = lo + kb * 16;
      if (pg < 0 || pg >= p.num_pages) {  // page of token t0 + (lane % 16), validated
        flag_bad(p.status, kSiteDecodeTable);
        pg = 0;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int tk = gq + 8 * u;
        const int page = __shfl_sync(0xffffffffu, pg, tk);
        const int t = t0 + tk;
        const __nv_bfloat16* row =
            p.kc + (static_cast<int64_t>(page) * P + (t % P)) * row_stride + static_cast<int64_t>(kvh) * kDecD;
#pragma unroll
        for (int c2 = 0; c2 < 4; ++c2) cp_async16(dst + (4 * u + c2) * 32, row + 32 * c2 + 8 * qq, t < hi ? 16 : 0);
      }
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int tv = 2 * qq + (w & 1) + 8 * (w >> 1);
        const int page = __shfl_sync(0xffffffffu, pg, tv);
        const int t = t0 + tv;
        const __nv_bfloat16* row =
            p.vc + (static_cast<int64_t>(page) * P + (t % P)) * row_stride + static_cast<int64_t>(kvh) * kDecD;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) cp_async16(dst + (8 + 2 * w + h2) * 32, row + 16 * gq + 8 * h2, t < hi ? 16 : 0);
      }
    }
    cp_async_commit();  // one group per call, empty past the last block
  };
  const int nmine = nblk > warp ? (nblk - warp + kDecWarps - 1) / kDecWarps : 0;
#pragma unroll
  for (int i = 0; i < kDecStages - 1; ++i) issue(warp + kDecWarps * i, i, page_entry(warp + kDecWarps * i));
  int pg_next = page_entry(warp + kDecWarps * (kDecStages - 1));

  for (int i = 0; i < nmine; ++i) {
    const int kb = warp + kDecWarps * i;
    const int t0 = lo + kb * 16;
    // keep kDecStages - 1 blocks in flight: the slot refilled held block i - 1
    issue(warp + kDecWarps * (i + kDecStages - 1), (i + kDecStages - 1) % kDecStages, pg_next);
    pg_next = page_entry(warp + kDecWarps * (i + kDecStages));
    cp_async_wait<kDecStages - 1>();  // block i has landed
    const uint4* src = my_ring + (i % kDecStages) * 16 * 32 + lane;
    uint4 kr[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int c2 = 0; c2 < 4; ++c2) kr[u][c2] = src[(4 * u + c2) * 32];
    uint4 vr[4][2];
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) vr[w][h2] = src[(8 + 2 * w + h2) * 32];

    // S = Q K^T for 16 tokens (two n-tiles of 8)
    float sc[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      sc[u][0] = sc[u][1] = sc[u][2] = sc[u][3] = 0.f;
#pragma unroll
      for (int cs = 0; cs < 8; ++cs) {
        const uint4 v = kr[u][cs >> 1];
        const uint32_t b0 = (cs & 1) ? v.z : v.x;
        const uint32_t b1 = (cs & 1) ? v.w : v.y;
        mma16816(sc[u], qa[cs], b0, b1);
      }
    }
    // mask tokens past the split end, and past each row's causal limit
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = t0 + 8 * u + 2 * qq + e;
        if (t >= lim0) sc[u][e] = -INFINITY;
        if (t >= lim1) sc[u][2 + e] = -INFINITY;
      }

    // online softmax, row g (and g+8 when both halves are in use); a row that
    // has seen no visible key yet (max -inf) shifts by 0 and keeps P = 0
    float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    const float mn0 = fmaxf(m0, mx0 * p.scale_log2);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
    const float al0 = ptx::ex2(m0 - mu0);
    m0 = mn0;
    float pr[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      pr[u][0] = ptx::ex2(fmaf(sc[u][0], p.scale_log2, -mu0));
      pr[u][1] = ptx::ex2(fmaf(sc[u][1], p.scale_log2, -mu0));
    }
    l0 = l0 * al0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
    float al1 = 1.f;
    if (kTwoRowHalves) {
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn1 = fmaxf(m1, mx1 * p.scale_log2);
      const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
      al1 = ptx::ex2(m1 - mu1);
      m1 = mn1;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        pr[u][2] = ptx::ex2(fmaf(sc[u][2], p.scale_log2, -mu1));
        pr[u][3] = ptx::ex2(fmaf(sc[u][3], p.scale_log2, -mu1));
      }
      l1 = l1 * al1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
    } else {
#pragma unroll
      for (int u = 0; u < 2; ++u) pr[u][2] = pr[u][3] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      acc[j][0] *= al0;
      acc[j][1] *= al0;
      if (kTwoRowHalves) {
        acc[j][2] *= al1;
        acc[j][3] *= al1;
      }
    }
    // P as the A operand (k = 16 tokens)
    uint32_t pa[4];
    pa[0] = ptx::pack_bf16(pr[0][0], pr[0][1]);
    pa[1] = ptx::pack_bf16(pr[0][2], pr[0][3]);
    pa[2] = ptx::pack_bf16(pr[1][0], pr[1][1]);
    pa[3] = ptx::pack_bf16(pr[1][2], pr[1][3]);
    // O += P V over the 16 n-tiles of the (permuted) head dimension
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int wd = j >> 1;  // 32-bit word within the 16-element chunk
      const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
      auto word = [&](int w) -> uint32_t {
        const uint4 x = vr[w][wd >> 2];
        const int k = wd & 3;
        return k == 0 ? x.x : (k == 1 ? x.y : (k == 2 ? x.z : x.w));
      };
      const uint32_t b0 = __byte_perm(word(0), word(1), sel);
      const uint32_t b1 = __byte_perm(word(2), word(3), sel);
      mma16816(acc[j], pa, b0, b1);
    }
  }

  // row sums across the quad
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  cp_async_wait<0>();
  __syncthreads();  // every warp is done with the ring before it holds the partials
  // per-warp partials to shared memory (un-permuting the head dimension)
  if (gq < nrows) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      s_o[warp][gq][16 * (2 * qq) + j] = acc[j][0];
      s_o[warp][gq][16 * (2 * qq + 1) + j] = acc[j][1];
    }
    if (qq == 0) {
      s_m[warp][gq] = m0;
      s_l[warp][gq] = l0;
    }
  }
  if (kTwoRowHalves && gq + 8 < nrows) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      s_o[warp][gq + 8][16 * (2 * qq) + j] = acc[j][2];
      s_o[warp][gq + 8][16 * (2 * qq + 1) + j] = acc[j][3];
    }
    if (qq == 0) {
      s_m[warp][gq + 8] = m1;
      s_l[warp][gq + 8] = l1;
    }
  }
  __syncthreads();

  // merge the four warps; thread -> (row, 4 columns)
  constexpr float kLn2 = 0.6931471805599453f;
  for (int idx = threadIdx.x; idx < nrows * (kDecD / 4); idx += blockDim.x) {
    const int r = idx / (kDecD / 4);
    const int c4 = (idx % (kDecD / 4)) * 4;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, s_m[w][r]);
    float o4[4] = {0.f, 0.f, 0.f, 0.f};
    float Lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float f = ptx::ex2(s_m[w][r] - M);
        Lsum += s_l[w][r] * f;
#pragma unroll
        for (int e = 0; e < 4; ++e) o4[e] += s_o[w][r][c4 + e] * f;
      }
    }
    // partial row (s, b, token r / G, head kvh * G + r % G)
    const int64_t row = ((static_cast<int64_t>(s) * p.batch + b) * QL + r / G) * p.hq + static_cast<int64_t>(kvh) * G +
                        r % G;
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    float4 out = make_float4(o4[0] * inv, o4[1] * inv, o4[2] * inv, o4[3] * inv);
    *reinterpret_cast<float4*>(p.part_o + row * kDecD + c4) = out;
    if (c4 == 0) p.part_lse[row] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
  }
}

// ------------------------------------------------------------------ launchers

template <int G>
static cudaError_t launch_split(bool two, dim3 grid, const DecodeParams& p, cudaStream_t stream) {
  if constexpr (G == 16) {
    return launch_after(decode_split_kernel<16, true>, grid, dim3(128), kDecRingBytes, stream, p);
  } else {
    if (two) return launch_after(decode_split_kernel<G, true>, grid, dim3(128), kDecRingBytes, stream, p);
    return launch_after(decode_split_kernel<G, false>, grid, dim3(128), kDecRingBytes, stream, p);
  }
}

cudaError_t launch_decode_general(const DecodeLaunch& a, float* part_o, float* part_lse, int32_t* status,
                                  cudaStream_t stream) {
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  p.vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  p.page_table = a.page_table;
  p.seqlens = a.seqlens_k;
  p.batch = a.batch;
  p.hq = a.q_heads;
  p.hkv = a.kv_heads;
  p.page_size = a.page_size;
  p.num_pages = a.num_pages;
  p.max_pages = a.max_pages;
  p.num_splits = a.num_splits;
  p.q_len = a.q_len;
  p.min_split = a.min_split_tokens;
  p.counts_out = a.split_counts_out;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.bounds_out = a.split_bounds_out;
  p.status = status;
  const int G = a.q_heads / a.kv_heads;
  const bool two = G * a.q_len > 8;
  dim3 grid(a.num_splits, a.kv_heads, a.batch);
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t ea = once_per_device(attr_done, [] {
    for (auto k : {decode_split_kernel<1, false>, decode_split_kernel<2, false>, decode_split_kernel<4, false>,
                   decode_split_kernel<8, false>, decode_split_kernel<1, true>, decode_split_kernel<2, true>,
                   decode_split_kernel<4, true>, decode_split_kernel<8, true>, decode_split_kernel<16, true>}) {
      const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecRingBytes);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  });
  if (ea != cudaSuccess) return ea;
  cudaEvent_t* ev = static_cast<cudaEvent_t*>(a.main_kernel_events);
  if (ev) cudaEventRecord(ev[0], stream);
  cudaError_t e;
  switch (G) {
    case 1: e = launch_split<1>(two, grid, p, stream); break;
    case 2: e = launch_split<2>(two, grid, p, stream); break;
    case 4: e = launch_split<4>(two, grid, p, stream); break;
    case 8: e = launch_split<8>(two, grid, p, stream); break;
    case 16: e = launch_split<16>(two, grid, p, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (ev) cudaEventRecord(ev[1], stream);
  if (e != cudaSuccess) return e;
  const int rows = a.batch * a.q_len * a.q_heads;  // (b, token, head) rows of O
  return launch_after(decode_merge_kernel, dim3((rows + 3) / 4), dim3(128), 0, stream, static_cast<const float*>(part_o),
                          static_cast<const float*>(part_lse), a.num_splits, rows, static_cast<__nv_bfloat16*>(a.o),
                          a.lse);
}

cudaError_t launch_decode(const jfa_decode_args& a, float* part_o, float* part_lse, int32_t* status,
                          cudaStream_t stream) {
  DecodeLaunch d;
  d.q = a.q;
  d.k_cache = a.k_cache;
  d.v_cache = a.v_cache;
  d.page_table = a.page_table;
  d.seqlens_k = a.seqlens_k;
  d.batch = a.batch;
  d.q_len = 1;
  d.q_heads = a.q_heads;
  d.kv_heads = a.kv_heads;
  d.page_size = a.page_size;
  d.num_pages = a.num_pages;
  d.max_pages = a.max_pages;
  d.num_splits = a.num_splits;
  d.min_split_tokens = 0;
  d.scale = a.scale;
  d.o = a.o;
  d.lse = a.lse;
  d.split_bounds_out = a.split_bounds_out;
  d.split_counts_out = nullptr;
  d.main_kernel_events = a.main_kernel_events;
  return launch_decode_general(d, part_o, part_lse, status, stream);
}

}  // namespace jfa
