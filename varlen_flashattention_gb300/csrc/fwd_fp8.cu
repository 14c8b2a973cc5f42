// Jagged FlashAttention forward with FP8 (e4m3) inputs, head_dim 128.
//
// "Optimizing FlashAttention-4 for Efficient Inference" (hpjadul), section
// "PR 2109: Support FP8 Inputs": the inference forward takes FP8 inputs, for
// less memory traffic and faster tensor-core math than bf16. The page gives
// no scale convention; here each of Q, K, V carries one descale factor (a
// byte x stands for e4m3(x) * descale), O is bf16 and LSE fp32, as in jfa_fwd.
//
// Same flat-stream schedule as the bf16 forward for head_dim 128
// (fwd_stream.cu): a persistent CTA runs its items of the longest-first queue
// as one stream of steps, S of the next step issued before P V of the current
// one, O double-buffered in TMEM, eight softmax warps (two per row, one per
// half of the keys) and four epilogue warps. What changes with 8-bit inputs:
//  * S = Q K^T and O += P V are tcgen05 MMAs of kind::f8f6f4 (K = 32 per
//    instruction); a 128 x 128 tile is 16 KB and one 128-byte swizzle row
//    holds a whole 128-element row, so Q, K and P stay K-major exactly as the
//    bf16 tiles do;
//  * O += P V needs V with the keys contiguous (the K-major B operand). A
//    pre-pass writes every 128-key tile of V transposed into its own
//    [head_dim x 128 keys] block (keys past the sequence zeroed), so each
//    block starts at x = 0 and every TMA start is 16-byte aligned;
//  * P (e4m3) goes to shared memory in the 128B-swizzled layout instead of
//    over S in TMEM, so the two softmax groups need no hand-off on S; its two
//    buffers follow the two score buffers (the MMA that reads P(x) completes
//    before S(x + 2) is issued, and the softmax waits for S(x + 2) before
//    writing P(x + 2) into the same buffer);
//  * scores are scaled by scale * q_descale * k_descale; O by v_descale / l.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "jfa_internal.h"
#include "ptx.cuh"
#include "trace.cuh"

namespace jfa {

namespace {

// Instruction descriptor, kind::f8f6f4 with e4m3 A and B (format code 0 in
// bits 7-9 and 10-12), fp32 accumulation, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], 8-bit inputs (K = 32 per instruction)
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

constexpr int kF8D = 128;                 // head_dim
constexpr int kF8TileBytes = kTile * kF8D;  // one 128 x 128 e4m3 tile

constexpr int kF8Threads = 448;  // warps 0-7 softmax, 8-11 epilogue, 12 TMA producer, 13 MMA issuer

struct Fp8Params {
  const int4* items;     // (b, h, query tile, key tiles)
  const int4* item_seq;  // (first row, length, first key-tile index, 0)
  int32_t* status;
  __nv_bfloat16* o;
  float* lse;
  int32_t heads, total;
  float s_log2;     // scale * q_descale * k_descale * log2(e)
  float v_descale;
  uint64_t budget_ns;
};

struct Fp8Layout {
  static constexpr int kQSlots = 2;
  static constexpr int kSlots = 6;                                  // K and V^T tiles
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = kQSlots * kF8TileBytes;
  static constexpr int kOffP = kOffSlots + kSlots * kF8TileBytes;  // two P buffers (e4m3)
  static constexpr int kOffOStage = kOffP + 2 * kF8TileBytes;       // O of a finished item (bf16, TMA store)
  static constexpr int kOffMl = kOffOStage + kTile * kF8D * 2;      // float2 (m, l) per row, two buffers
  static constexpr int kOffBars = kOffMl + 2 * kTile * 8;
  // q_full[2], q_empty[2], slot_full[S], slot_empty[S], s_full[2], p_full[2], o_ready[2], o_final[2],
  // o_free[2], ml_half[2], ml_full[2], ml_empty[2], drain, o_staged, o_stage_read
  static constexpr int kNumBars = 2 * kQSlots + 2 * kSlots + 9 * 2 + 3 + 16;  // + half_max[2][2][4]
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;  // slack for the 1024-byte alignment of the tiles
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384, kTmemCols = 512;
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// One 32-bit TMEM column of this warp's 32 lanes.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t v;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr) : "memory");
  return v;
}

struct Fp8Item {
  int h, t;
  int q_row, kv_row0, L, n_kv, vt0;
  int64_t lse0;
};

__device__ __forceinline__ Fp8Item fp8_item(const Fp8Params& p, int idx) {
  const int4 it = p.items[idx];
  const int4 sq = p.item_seq[idx];
  Fp8Item I;
  I.h = it.y;
  I.t = it.z;
  I.n_kv = it.w;  // the queue's cost of a forward item: key tiles visited
  I.kv_row0 = sq.x;
  I.L = sq.y;
  I.vt0 = sq.z;  // the sequence's first tile index: its key tile j is V^T block vt0 + j
  I.q_row = sq.x + kTile * I.t;
  I.lse0 = static_cast<int64_t>(I.h) * p.total + I.q_row;
  return I;
}

// Load order (and consumption order): Q of an item, then K of its first step;
// for every step j, K of step j + 1 (or the next item's Q and first K) before
// V of step j.
template <class FQ, class FK, class FV>
__device__ __forceinline__ void fp8_walk_loads(const Fp8Params& p, int first, int stride, int n_items, FQ on_q,
                                               FK on_k, FV on_v) {
  if (first >= n_items) return;
  Fp8Item cur = fp8_item(p, first), nxt;
  if (!on_q(cur) || !on_k(cur, 0)) return;
  for (int idx = first; idx < n_items; idx += stride) {
    const bool more = idx + stride < n_items;
    if (more) nxt = fp8_item(p, idx + stride);
    for (int j = 0; j < cur.n_kv; ++j) {
      if (j + 1 < cur.n_kv) {
        if (!on_k(cur, j + 1)) return;
      } else if (more) {
        if (!on_q(nxt) || !on_k(nxt, 0)) return;
      }
      if (!on_v(cur, j)) return;
    }
    cur = nxt;
  }
}

// The flat-stream forward of fwd_stream.cu with 8-bit operands. Every item of
// the self-attention queue has at least one key tile.
template <bool CAUSAL>
__global__ void __launch_bounds__(kF8Threads, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_vt, const __grid_constant__ CUtensorMap tm_o,
                   const Fp8Params p) {
  using Lay = Fp8Layout;
  constexpr int kSlots = Lay::kSlots;
  constexpr int kQS = Lay::kQSlots;
  constexpr uint32_t kIdesc = idesc_e4m3(128, 128);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBars);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + kQS;
  uint64_t* slot_full = q_empty + kQS;
  uint64_t* slot_empty = slot_full + kSlots;
  uint64_t* s_full = slot_empty + kSlots;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_ready = p_full + 2;
  uint64_t* o_final = o_ready + 2;
  uint64_t* o_free = o_final + 2;
  uint64_t* ml_half = o_free + 2;
  uint64_t* ml_full = ml_half + 2;
  uint64_t* ml_empty = ml_full + 2;
  uint64_t* half_max = ml_empty + 2;  // [S buffer][group][warp quarter]: the group's row maxima are published
  uint64_t* drain = half_max + 16;
  uint64_t* o_staged = drain + 1;      // every epilogue thread has written its row of the O staging
  uint64_t* o_stage_read = drain + 2;  // the TMA store of the previous staged O has read it
  float2* ml = reinterpret_cast<float2*>(smem + Lay::kOffMl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  ptx::CtaCtl* ctl = reinterpret_cast<ptx::CtaCtl*>(smem + Lay::kOffMisc + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQS; ++i) {
      ptx::mbar_init(q_full + i, 1);
      ptx::mbar_init(q_empty + i, 1);
    }
    for (int i = 0; i < kSlots; ++i) {
      ptx::mbar_init(slot_full + i, 1);
      ptx::mbar_init(slot_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(s_full + i, 1);
      ptx::mbar_init(p_full + i, 8);  // the eight softmax warps
      ptx::mbar_init(o_ready + i, 1);
      ptx::mbar_init(o_final + i, 1);
      ptx::mbar_init(o_free + i, 4);       // the four epilogue warps
      ptx::mbar_init(ml_half + i, kTile);  // every group-0 softmax thread
      ptx::mbar_init(ml_full + i, kTile);  // every group-1 softmax thread
      ptx::mbar_init(ml_empty + i, 4);     // the four epilogue warps
    }
    for (int i = 0; i < 16; ++i) ptx::mbar_init(half_max + i, 1);  // one softmax warp each
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(o_staged, kTile);
    ptx::mbar_init(o_stage_read, 1);
    ctl->abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 12 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_vt);
    ptx::prefetch_tmap(&tm_o);
  }
  __syncthreads();
  if (warp == 13) {
    ptx::tmem_alloc(tmem_slot, Lay::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  wait_prior_grid();  // the set-up above is local; the queue's items are read below
  const uint32_t tmem = *tmem_slot;
  const int n_items = p.status[2];
  int32_t* status = p.status;
  const uint64_t budget = p.budget_ns;
  const int cta = blockIdx.x, n_ctas = gridDim.x;

  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t pos = 0, kq = 0;
      auto on_kv = [&](const CUtensorMap* map, int x, int y) -> bool {
        const uint32_t slot = pos % kSlots, round = pos / kSlots;
        if (!ptx::mbar_wait(slot_empty + slot, (round & 1) ^ 1, ctl, status, kSiteFwdProdSlot, budget)) return false;
        ptx::mbar_arrive_expect_tx(slot_full + slot, kF8TileBytes);
        ptx::tma_load_2d(smem + Lay::kOffSlots + slot * kF8TileBytes, map, slot_full + slot, x, y);
        ++pos;
        return true;
      };
      auto on_q = [&](const Fp8Item& I) -> bool {
        // debug builds: the Q tile and every K/V tile start inside their sequences and heads
        if (!JFA_TILE_OK(I.t >= 0 && kTile * I.t < I.L && I.h >= 0 && I.h < p.heads, ctl, status, kSiteCheckFwdQ))
          return false;
        if (!JFA_TILE_OK(I.n_kv > 0 && kTile * (I.n_kv - 1) < I.L && I.vt0 >= 0, ctl, status, kSiteCheckFwdKV))
          return false;
        const uint32_t qs = kq % kQS, qround = kq / kQS;
        if (!ptx::mbar_wait(q_empty + qs, (qround & 1) ^ 1, ctl, status, kSiteFwdProdQ, budget)) return false;
        ptx::mbar_arrive_expect_tx(q_full + qs, kF8TileBytes);
        ptx::tma_load_2d(smem + Lay::kOffQ + qs * kF8TileBytes, &tm_q, q_full + qs, I.h * kF8D, I.q_row);
        ++kq;
        return true;
      };
      fp8_walk_loads(
          p, cta, n_ctas, n_items, on_q,
          [&](const Fp8Item& I, int j) { return on_kv(&tm_k, I.h * kF8D, I.kv_row0 + kTile * j); },
          [&](const Fp8Item& I, int j) { return on_kv(&tm_vt, 0, ((I.vt0 + j) * p.heads + I.h) * kF8D); });
      // an aborted pipeline may leave fills without a consumer: wait (bounded) for them
      ptx::CtaCtl no_abort{0, 0};
      for (uint32_t i = pos > kSlots ? pos - kSlots : 0; i < pos; ++i)
        ptx::mbar_wait(slot_full + i % kSlots, (i / kSlots) & 1, &no_abort, nullptr, kSiteFwdDrain, budget);
      for (uint32_t i = kq > kQS ? kq - kQS : 0; i < kq; ++i)
        ptx::mbar_wait(q_full + i % kQS, (i / kQS) & 1, &no_abort, nullptr, kSiteFwdDrain, budget);
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop; one elected lane issues each group of MMAs.
    uint32_t pos = 0;
    bool ok = true;
    auto slot_wait = [&](uint32_t& slot) -> bool {
      slot = pos % kSlots;
      const bool w = ptx::mbar_wait(slot_full + slot, (pos / kSlots) & 1, ctl, status, kSiteFwdMmaSlot, budget);
      ptx::tc_fence_after();
      ++pos;
      return ptx::warp_all(w);
    };
    auto q_wait = [&](uint32_t kq) -> bool {
      const bool w = ptx::mbar_wait(q_full + kq % kQS, (kq / kQS) & 1, ctl, status, kSiteFwdMmaQ, budget);
      ptx::tc_fence_after();
      return ptx::warp_all(w);
    };
    // S(x) = Q K^T into S buffer x & 1: 4 MMAs of K = 32; last_q_use releases the Q buffer
    auto issue_s = [&](uint32_t kq, uint32_t x, bool last_q_use) -> bool {
      uint32_t slot;
      if (!slot_wait(slot)) return false;
      const uint32_t qs = kq % kQS;
      const uint32_t q_addr = ptx::smem_u32(smem + Lay::kOffQ + qs * kF8TileBytes);
      const uint32_t k_addr = ptx::smem_u32(smem + Lay::kOffSlots + slot * kF8TileBytes);
      const uint32_t d_tmem = tmem + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kF8D / 32; ++kk)
          mma_ss_f8(d_tmem, ptx::sdesc_sw128(q_addr + kk * 32, 16, 1024), ptx::sdesc_sw128(k_addr + kk * 32, 16, 1024),
                    kIdesc, kk > 0 ? 1u : 0u);
        ptx::mma_commit(s_full + (x & 1));
        ptx::mma_commit(slot_empty + slot);
        if (last_q_use) ptx::mma_commit(q_empty + qs);
      }
      __syncwarp();
      return true;
    };
    int idx = cta;
    Fp8Item cur, nxt;
    if (idx < n_items) cur = fp8_item(p, idx);
    uint32_t kq = 0, x = 0;  // items so far, steps so far
    if (idx < n_items) ok = q_wait(0) && issue_s(0, 0, cur.n_kv == 1);
    while (ok && idx < n_items) {
      const int nidx = idx + n_ctas;
      const bool more = nidx < n_items;
      if (more) nxt = fp8_item(p, nidx);
      const int n = cur.n_kv;
      const uint32_t ob = kq & 1;
      for (int j = 0; ok && j < n; ++j, ++x) {
        if (j + 1 < n) {
          if (!(ok = issue_s(kq, x + 1, j + 2 == n))) break;
        } else if (more) {
          if (!(ok = q_wait(kq + 1) && issue_s(kq + 1, x + 1, nxt.n_kv == 1))) break;
        }
        uint32_t slot;
        if (!(ok = slot_wait(slot))) break;  // V^T of this step
        bool w = true;
        if (j == 0 && kq >= 2)  // the epilogue of item kq - 2 has read this O buffer
          w = ptx::mbar_wait(o_free + ob, ((kq - 2) >> 1) & 1, ctl, status, kSiteFwdMmaOFree, budget);
        w = w && ptx::mbar_wait(p_full + (x & 1), (x >> 1) & 1, ctl, status, kSiteFwdMmaP, budget);
        if (!(ok = ptx::warp_all(w))) break;
        ptx::tc_fence_after();
        const uint32_t vt_addr = ptx::smem_u32(smem + Lay::kOffSlots + slot * kF8TileBytes);
        const uint32_t p_addr = ptx::smem_u32(smem + Lay::kOffP + (x & 1) * kF8TileBytes);
        const uint32_t o_tmem = tmem + (ob ? Lay::kColO1 : Lay::kColO0);
        if (ptx::elect_one()) {
          // O += P V: A = P in shared memory, B = the V^T block, both K-major over the keys
#pragma unroll
          for (int kk = 0; kk < kTile / 32; ++kk)
            mma_ss_f8(o_tmem, ptx::sdesc_sw128(p_addr + kk * 32, 16, 1024),
                      ptx::sdesc_sw128(vt_addr + kk * 32, 16, 1024), kIdesc, (j > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(o_ready + (x & 1));
          ptx::mma_commit(slot_empty + slot);
          if (j + 1 == n) ptx::mma_commit(o_final + ob);
        }
        __syncwarp();
      }
      ++kq;
      cur = nxt;
      idx = nidx;
    }
    if (ptx::elect_one()) ptx::mma_commit(drain);
    __syncwarp();
    ptx::CtaCtl no_abort{0, 0};
    ptx::mbar_wait(drain, 0, &no_abort, nullptr, kSiteFwdDrain, budget);
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax (warps 0-7)
    // Two warps per row: group g exponentiates key columns 64 g .. 64 g + 63;
    // both read the whole row for the maximum, so they rescale alike. P goes
    // to shared memory, so no group overwrites scores the other still reads.
    const int g = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int c_own = 64 * g, c_other = 64 - c_own;
    const float sl = p.s_log2;
    uint8_t* p_row = smem + Lay::kOffP + r * 128;  // this row in P buffer 0 (buffer 1: + 16 KB)
    const int sw = r & 7;
    uint32_t x = 0, kq = 0;
    bool ok = true, s_ready = false;
    Fp8Item nxt;
    if (cta < n_items) nxt = fp8_item(p, cta);
    for (int idx = cta; ok && idx < n_items; idx += n_ctas) {
      const Fp8Item I = nxt;
      if (idx + n_ctas < n_items) nxt = fp8_item(p, idx + n_ctas);
      const int n = I.n_kv;
      const uint32_t ob = kq & 1;
      const uint32_t o_tmem = tmem + lane_base + (ob ? Lay::kColO1 : Lay::kColO0) + c_own;
      const int qi = kTile * I.t + r;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j, ++x) {
        const uint32_t s_tmem = tmem + lane_base + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
        if (!s_ready && !(ok = ptx::mbar_wait(s_full + (x & 1), (x >> 1) & 1, ctl, status, kSiteFwdSoftS, budget)))
          break;
        ptx::tc_fence_after();
        const int lim = CAUSAL ? min(qi + 1 - kTile * j, I.L - kTile * j) : I.L - kTile * j;
        auto mask = [&](uint32_t(&v)[32], int c0) {
          if (lim < c0 + 32) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c0 + e >= lim) v[e] = __float_as_uint(-INFINITY);
          }
        };
        // this group's half of the row (it stays in registers) and its maximum
        uint32_t sa[2][32];
        ptx::tmem_ld32(s_tmem + c_own, sa[0]);
        ptx::tmem_ld32(s_tmem + c_own + 32, sa[1]);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(sa[0]);
        ptx::reg_fence32(sa[1]);
        mask(sa[0], c_own);
        mask(sa[1], c_own + 32);
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            mx8[(e >> 1) & 7] = ptx::fmax3(mx8[(e >> 1) & 7], __uint_as_float(sa[u][e]), __uint_as_float(sa[u][e + 1]));
        const float hmax = fmaxf(ptx::fmax3(mx8[0], mx8[1], mx8[2]),
                                 ptx::fmax3(ptx::fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        // The halves' maxima are exchanged through the last TMEM column of each
        // half (read into registers already; P goes to shared memory); after an
        // item's first step the exponentials run against the running max before
        // the other half's maximum is known, and again only if it grew by > 2^8.
        tmem_st1(s_tmem + c_own + 63, __float_as_uint(hmax));
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(half_max + ((x & 1) * 2 + g) * 4 + quarter);
        uint64_t* other = half_max + ((x & 1) * 2 + (1 - g)) * 4 + quarter;
        auto other_max = [&]() -> float {  // after `other` has completed
          ptx::tc_fence_after();
          const uint32_t v = tmem_ld1(s_tmem + c_other + 63);
          ptx::tmem_ld_wait();
          return __uint_as_float(v);
        };
        // P = 2^(S sl - m) as e4m3: this group's 64 keys, 16 per 16-byte chunk of
        // the swizzled row; returns the half-row sum
        uint8_t* prow = p_row + (x & 1) * kF8TileBytes;
        const uint64_t sl2 = ptx::f2_packf(sl, sl);
        auto exps = [&](float mref) -> float {
          const float mu = (mref == -INFINITY) ? 0.f : mref;
          const uint64_t nmu2 = ptx::f2_packf(-mu, -mu);
          uint64_t ls2[2] = {ptx::f2_packf(0.f, 0.f), ptx::f2_packf(0.f, 0.f)};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {  // keys 4 e .. 4 e + 3 of this 32-key half
              float q0, q1, q2, q3;
              ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(sa[u][4 * e], sa[u][4 * e + 1]), sl2, nmu2), q0, q1);
              ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(sa[u][4 * e + 2], sa[u][4 * e + 3]), sl2, nmu2), q2, q3);
              const float p0 = ptx::ex2(q0), p1 = ptx::ex2(q1), p2 = ptx::ex2(q2), p3 = ptx::ex2(q3);
              ls2[e & 1] = ptx::f2_add(ls2[e & 1], ptx::f2_add(ptx::f2_packf(p0, p1), ptx::f2_packf(p2, p3)));
              const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE, __NV_E4M3);
              const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(p2, p3), __NV_SATFINITE, __NV_E4M3);
              w[e] = lo | (hi << 16);
            }
            const int ch = (c_own >> 4) + 2 * u;  // 16-byte chunks ch, ch + 1 of the 128-byte row
            ptx::st_shared_v4(prow + ((ch ^ sw) << 4), w[0], w[1], w[2], w[3]);
            ptx::st_shared_v4(prow + (((ch + 1) ^ sw) << 4), w[4], w[5], w[6], w[7]);
          }
          float a0, a1, b0, b1;
          ptx::f2_unpack(ls2[0], a0, a1);
          ptx::f2_unpack(ls2[1], b0, b1);
          return (a0 + a1) + (b0 + b1);
        };
        float lsum = 0.f;
        if (j == 0) {
          if (!(ok = ptx::mbar_wait(other, (x >> 1) & 1, ctl, status, kSiteFwdSoftS, budget))) break;
          m = fmaxf(hmax, other_max()) * sl;
          lsum = exps(m);
        } else {
          lsum = exps(m);
          if (!(ok = ptx::mbar_wait(other, (x >> 1) & 1, ctl, status, kSiteFwdSoftS, budget))) break;
          const float mnew = fmaxf(hmax, other_max()) * sl;
          // rescale O only when the row max grows by more than 2^8 (P stays below 2^8 < 448)
          const bool need = mnew > m + 8.0f;
          if (__any_sync(0xffffffffu, need)) {
            const float mm = need ? mnew : m;
            const float f = ptx::ex2(m - mm);
            const uint32_t xp = x - 1;
            if (!(ok = ptx::mbar_wait(o_ready + (xp & 1), (xp >> 1) & 1, ctl, status, kSiteFwdSoftO, budget)))
              break;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {  // this group's 64 columns of O, 16 at a time
              uint32_t ov[16];
              ptx::tmem_ld16(o_tmem + 16 * c, ov);
              ptx::tmem_ld_wait();
              ptx::reg_fence16(ov);
#pragma unroll
              for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
              ptx::tmem_st16(o_tmem + 16 * c, ov);
            }
            ptx::tmem_st_wait();
            l *= f;
            m = mm;
            lsum = exps(m);  // again, against the new reference (over the first try's P)
          }
        }
        l += lsum;
        if (j + 1 == n) {
          // row statistics of the finished item: group 0 stores (m, its sum), group 1 adds its sum
          if (g == 0) {
            if (kq >= 2 &&
                !(ok = ptx::mbar_wait(ml_empty + ob, ((kq - 2) >> 1) & 1, ctl, status, kSiteFwdSoftMl, budget)))
              break;
            ml[ob * kTile + r] = make_float2(m, l);
            ptx::mbar_arrive(ml_half + ob);
          } else {
            if (!(ok = ptx::mbar_wait(ml_half + ob, (kq >> 1) & 1, ctl, status, kSiteFwdSoftMl, budget))) break;
            ml[ob * kTile + r].y += l;
            ptx::mbar_arrive(ml_full + ob);
          }
        }
        s_ready = ptx::mbar_test(s_full + ((x + 1) & 1), ((x + 1) >> 1) & 1);
        ptx::fence_proxy_async_smem();  // the tensor core reads P through the async proxy
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full + (x & 1));
      }
      ++kq;
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 8-11)
    // O * v_descale / l of whole query tiles leaves by TMA store through a bf16
    // staging buffer (128B swizzle, two 64-column atoms); partial tiles row by row.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr float kLn2 = 0.6931471805599453f;
    const bool issuer = warp == 8 && lane == 0;
    uint8_t* ostage = smem + Lay::kOffOStage;
    uint32_t kq = 0, n_st = 0;
    Fp8Item nxt;
    if (cta < n_items) nxt = fp8_item(p, cta);
    for (int idx = cta; idx < n_items; idx += n_ctas) {
      const Fp8Item I = nxt;
      if (idx + n_ctas < n_items) nxt = fp8_item(p, idx + n_ctas);
      const bool row_ok = kTile * I.t + r < I.L;
      __nv_bfloat16* orow = p.o + (static_cast<int64_t>(I.q_row) + r) * p.heads * kF8D + static_cast<int64_t>(I.h) * kF8D;
      const uint32_t ob = kq & 1;
      bool w = ptx::mbar_wait(o_final + ob, (kq >> 1) & 1, ctl, status, kSiteFwdEpi, budget);
      w = w && ptx::mbar_wait(ml_full + ob, (kq >> 1) & 1, ctl, status, kSiteFwdEpi, budget);
      if (!w) break;
      ptx::tc_fence_after();
      const float2 st = ml[ob * kTile + r];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ml_empty + ob);
      const float f = st.y > 0.f ? p.v_descale / st.y : 0.f;
      const uint32_t o_tmem = tmem + lane_base + (ob ? Lay::kColO1 : Lay::kColO0);
      const bool staged = I.L - kTile * I.t >= kTile;
      if (staged && n_st > 0) {  // the previous TMA store has read the staging
        if (issuer) {
          ptx::bulk_wait_read0();
          ptx::mbar_arrive(o_stage_read);
        }
        if (!ptx::mbar_wait(o_stage_read, (n_st - 1) & 1, ctl, status, kSiteFwdEpi, budget)) break;
      }
#pragma unroll 1
      for (int c = 0; c < kF8D / 32; ++c) {
        uint32_t ov[32];
        ptx::tmem_ld32(o_tmem + 32 * c, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(ov);
        if (c == kF8D / 32 - 1) {  // all of O is in registers: the next item may use this buffer
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(o_free + ob);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            wv[e] = ptx::pack_bf16(__uint_as_float(ov[8 * q4 + 2 * e]) * f, __uint_as_float(ov[8 * q4 + 2 * e + 1]) * f);
          if (staged)
            ptx::st_shared_v4(ostage + (c >> 1) * 16384 + r * 128 + (((((c & 1) << 2) + q4) ^ (r & 7)) << 4), wv[0],
                              wv[1], wv[2], wv[3]);
          else if (row_ok)
            ptx::st_v4(orow + 32 * c + 8 * q4, wv[0], wv[1], wv[2], wv[3]);
        }
      }
      if (staged) {
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(o_staged);
        if (!ptx::mbar_wait(o_staged, n_st & 1, ctl, status, kSiteFwdEpi, budget)) break;
        if (issuer) {
          ptx::tma_store_2d(&tm_o, ostage, I.h * kF8D, I.q_row);
          ptx::tma_store_2d(&tm_o, ostage + 16384, I.h * kF8D + 64, I.q_row);
          ptx::bulk_commit();
        }
        ++n_st;
      }
      if (row_ok) p.lse[I.lse0 + r] = (st.x + log2f(st.y)) * kLn2;
      ++kq;
    }
    if (issuer) ptx::bulk_wait0();  // every O store has completed
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

// 4 x 4 byte transpose: a, b, c, d hold bytes 0-3 of four rows; w[j] gets
// byte j of each row, row order preserved.
__device__ __forceinline__ void transpose4x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t (&w)[4]) {
  const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(c, d, 0x5140);  // a0 b0 a1 b1, c0 d0 c1 d1
  const uint32_t t2 = __byte_perm(a, b, 0x7362), t3 = __byte_perm(c, d, 0x7362);  // a2 b2 a3 b3, c2 d2 c3 d3
  w[0] = __byte_perm(t0, t1, 0x5410);
  w[1] = __byte_perm(t0, t1, 0x7632);
  w[2] = __byte_perm(t2, t3, 0x5410);
  w[3] = __byte_perm(t2, t3, 0x7632);
}

// V (e4m3 [total, H, 128]; with QUANT, bf16 values quantized on the way to
// e4m3(v * inv_descale), round to nearest even, saturating at +-448) -> one
// [128 head-dim rows x 128 keys] block per key tile and head: block (g * H + h)
// holds key tile g (tile_base numbering) of head h, keys past the end of the
// sequence zero. In self-attention every
// query tile is also a key tile, so the forward queue's items (head, tile,
// sequence start and tile base) name the blocks; a few CTAs per SM walk them.
// Per item: the 16 KB tile is read from global memory whole rows at a time
// (lane l of a warp reads 16-byte chunk l % 8 of row l / 8 + 4 w + 32 m) into
// shared memory, chunk c of key row k at position c ^ (k / 4 % 8); then lane l
// of warp w takes keys 4 l .. 4 l + 3 at head-dim columns 16 w .. 16 w + 15
// (one 16-byte read per key, conflict-free under that swizzle), transposes
// 4 x 4 byte blocks in registers and writes 4 keys of 16 head-dim rows, so
// every warp store is one contiguous 128-byte row of the block. With QUANT a
// lane reads the 32 bf16 bytes behind its 16 output bytes and converts them.
constexpr int kVtThreads = 256;
template <bool QUANT>
__global__ void __launch_bounds__(kVtThreads) vt_transpose_kernel(const uint8_t* __restrict__ v, const int4* items,
                                                                  const int4* item_seq, const int32_t* status,
                                                                  int heads, float inv_descale,
                                                                  uint8_t* __restrict__ vt) {
  __shared__ __align__(16) uint8_t tile[kTile * kF8D];
  wait_prior_grid();
  allow_next_grid();
  if (status[0] != JFA_OK) return;
  const int n_items = status[2];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int idx = blockIdx.x; idx < n_items; idx += gridDim.x) {
    const int4 it = items[idx], sq = item_seq[idx];
    const int h = it.y, j = it.z;        // head, tile of the sequence
    const int s0 = sq.x, gt = sq.z + j;  // sequence start; tile index in tile_base numbering
    const int rows = min(kTile, sq.y - kTile * j);  // valid keys of the tile
    const int c = lane & 7;
    uint4 g[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int k = (lane >> 3) + 4 * w + 32 * m;
      g[m] = make_uint4(0, 0, 0, 0);
      if (k < rows) {
        const int64_t e0 = ((static_cast<int64_t>(s0) + kTile * j + k) * heads + h) * kF8D + 16 * c;  // element
        if constexpr (!QUANT) {
          g[m] = ptx::ld_nc_v4(v + e0);
        } else {
          const uint4 lo = ptx::ld_nc_v4(v + 2 * e0), hi = ptx::ld_nc_v4(v + 2 * e0 + 16);  // 16 bf16 values
          const uint32_t in[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
          uint32_t out[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t b[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t x = in[2 * q + u];  // two bf16: element 2 (2q + u) in the low half
              const float2 f = make_float2(__uint_as_float(x << 16) * inv_descale,
                                           __uint_as_float(x & 0xffff0000u) * inv_descale);
              b[u] = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);  // low byte: f.x
            }
            out[q] = b[0] | (b[1] << 16);
          }
          g[m] = make_uint4(out[0], out[1], out[2], out[3]);
        }
      }
    }
    __syncthreads();  // the previous item's reads of the tile are done
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int k = (lane >> 3) + 4 * w + 32 * m;
      *reinterpret_cast<uint4*>(tile + k * kF8D + ((c ^ ((k >> 2) & 7)) << 4)) = g[m];
    }
    __syncthreads();
    const int k0 = 4 * lane, d0 = 16 * w;
    uint4 r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = k0 + i;
      r[i] = *reinterpret_cast<const uint4*>(tile + k * kF8D + ((w ^ ((k >> 2) & 7)) << 4));
    }
    uint8_t* out = vt + (static_cast<int64_t>(gt) * heads + h) * kF8D * kTile + k0;
    auto word = [](const uint4& x, int q) { return q == 0 ? x.x : (q == 1 ? x.y : (q == 2 ? x.z : x.w)); };
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // head-dim columns d0 + 4 q .. d0 + 4 q + 3
      uint32_t t[4];
      transpose4x4(word(r[0], q), word(r[1], q), word(r[2], q), word(r[3], q), t);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        *reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(d0 + 4 * q + e) * kTile) = t[e];
    }
  }
}

template <bool CAUSAL>
cudaError_t launch_fp8_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const CUtensorMap& to,
                         const Fp8Params& p, int grid, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(fwd_fp8_kernel<CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Fp8Layout::kAlloc);
  });
  if (e != cudaSuccess) return e;
  return launch_after(fwd_fp8_kernel<CAUSAL>, dim3(grid), dim3(kF8Threads), Fp8Layout::kAlloc, stream, tq, tk, tvt, to,
                      p);
}

}  // namespace

cudaError_t launch_vt_transpose(const void* v, const int4* items, const int4* item_seq, const int32_t* status,
                                int heads, int max_items, void* vt, cudaStream_t stream, const float* inv_descale) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  const int grid = std::max(1, std::min(max_items, 8 * sms));  // a few blocks per SM walk the items
  if (inv_descale)
    return launch_after(vt_transpose_kernel<true>, dim3(grid), dim3(kVtThreads), 0, stream,
                        static_cast<const uint8_t*>(v), items, item_seq, static_cast<const int32_t*>(status), heads,
                        *inv_descale, static_cast<uint8_t*>(vt));
  return launch_after(vt_transpose_kernel<false>, dim3(grid), dim3(kVtThreads), 0, stream,
                      static_cast<const uint8_t*>(v), items, item_seq, static_cast<const int32_t*>(status), heads, 1.0f,
                      static_cast<uint8_t*>(vt));
}

cudaError_t launch_fwd_fp8(bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const CUtensorMap& to, const int4* items, const int4* item_seq, int32_t* status, void* o, float* lse, int heads,
                           int total, float s_log2, float v_descale, uint64_t budget_ns, int grid,
                           cudaStream_t stream) {
  Fp8Params p;
  p.items = items;
  p.item_seq = item_seq;
  p.status = status;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.heads = heads;
  p.total = total;
  p.s_log2 = s_log2;
  p.v_descale = v_descale;
  p.budget_ns = budget_ns;
  return causal ? launch_fp8_t<true>(tq, tk, tvt, to, p, grid, stream)
                : launch_fp8_t<false>(tq, tk, tvt, to, p, grid, stream);
}

}  // namespace jfa
