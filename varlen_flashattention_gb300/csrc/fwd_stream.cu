// Jagged FlashAttention forward as a flat stream of steps, head_dim 128.
//
// What it computes is the forward of fwd.cu ("Cutting-edge isn't
// plug-and-play: customizing FA4 on B300", FlashAttention recap; "Optimizing
// Jagged Flash Attention with TLX", third paragraph). The difference is how
// the work is scheduled. A persistent CTA takes items (one query tile of one
// sequence and head) from the longest-first queue and runs all of its items
// as one stream of steps (one step = one key/value tile of one item), so that
// nothing drains between items: the S = Q K^T of the next step is issued
// before the P V of the current one even when the next step belongs to the
// next item, O is double-buffered in TMEM (items alternate between the two
// accumulators), and separate epilogue warps normalise and store an item's O
// while the next item is computed.
//
// The softmax is the slow side of a step (128 exponentials per row against
// 16 MMAs of 128x128x16), so two warps share every row: warps 0-3 (group 0)
// exponentiate key columns 0-63 of the score tile and warps 4-7 (group 1)
// columns 64-127, each on its own TMEM lanes' quarter (warp w reads lanes
// 32 (w % 4) ..). Each group reads only its own half of the score row and
// publishes that half's maximum in the half's last TMEM column (one mbarrier
// per warp quarter, group and S buffer); the other group reads it there, so
// both reach the same row maximum and the same rescaling decision. Each
// writes its half of P (bf16 pairs) over the first 32 TMEM columns of its own
// half of S. Each group keeps the sum of its own half of the row; the two
// sums meet in shared memory at the end of an item.
//
// Roles (448 threads): warps 0-7 softmax, warps 8-11 epilogue, warp 12 TMA
// producer, warp 13 MMA issuer (the whole warp runs the loop, one elected
// lane issues).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "jfa_internal.h"
#include "ptx.cuh"
#include "trace.cuh"

namespace jfa {

namespace {

constexpr int kD2 = 128;
constexpr int kThreads = 448;

struct FwdStreamParams {
  const int4* items;     // (b, h, query tile, key tiles)
  const int4* item_seq;  // (first row, length, tile_base) of the item's key sequence
  int32_t* status;
  __nv_bfloat16* o;
  float* lse;
  int32_t heads, total, bcast, q_len;
  int32_t var, group;    // varlen: item_seq holds query and key bounds; query heads per KV head
  float scale_log2;
  uint64_t budget_ns;
  int32_t* counter;      // items handed out so far (zero at launch): the producers claim items from it
};

struct FwdStreamLayout {
  static constexpr int kQBytes = kTile * kD2 * 2;   // one query tile: 128 rows x 128 d
  static constexpr int kKVBytes = kTile * kD2 * 2;  // one K or V tile
  static constexpr int kQSlots = 2;
  static constexpr int kSlots = 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = kQSlots * kQBytes;
  static constexpr int kOffOStage = kOffSlots + kSlots * kKVBytes;  // O of a finished item (bf16, TMA store)
  static constexpr int kOffMl = kOffOStage + kTile * kD2 * 2;        // float2 (m, l) per row, two buffers
  static constexpr int kRing = 8;                                    // claimed items in flight
  static constexpr int kOffRing = kOffMl + 2 * kTile * 8;            // int4 pairs (item, item_seq) per entry
  static constexpr int kOffBars = kOffRing + kRing * 32;
  // q_full[2], q_empty[2], slot_full[S], slot_empty[S], s_full[2], p_full[2],
  // o_ready[2], o_final[2], o_free[2], ml_half[2], ml_full[2], ml_empty[2],
  // half_max[2][2][4], drain, o_staged, o_stage_read, ring_full[R], ring_empty[R]
  static constexpr int kNumBars = 2 * kQSlots + 2 * kSlots + 8 * 2 + 16 + 1 + 2 + 2 * kRing;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 32;
  // Tiles need 1024-byte alignment; the dynamic shared-memory base is
  // 1024-byte aligned on this part (a kernel that finds it otherwise reports
  // JFA_ERR_UNSUPPORTED), so no slack is reserved.
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384, kTmemCols = 512;
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(kOffRing % 16 == 0 && kOffBars % 8 == 0, "ring and barrier alignment");
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

struct FwdStreamItem {
  int b, h, t;
  int hk;     // KV head read by query head h
  int delta;  // L_k - L_q: key j is visible to query i iff j <= i + delta (causal)
  int q_tma_row, kv_row0, Lq, Lk, n_kv;
  int64_t o_row, lse0;
};

// An item's record: the queue's (b, h, tile, key tiles) and the item's
// sequence bounds, stored side by side, so nothing waits on a dependent load.
__device__ __forceinline__ FwdStreamItem item_from(const FwdStreamParams& p, int4 it, int4 sq) {
  FwdStreamItem I;
  I.b = it.x;
  I.h = it.y;
  I.t = it.z;
  const int s0 = sq.x;
  I.Lk = sq.y;
  I.kv_row0 = s0;
  I.hk = I.h;
  I.delta = 0;
  if (p.var) {  // (first query row, L_q, first key row, L_k)
    I.Lq = sq.y;
    I.kv_row0 = sq.z;
    I.Lk = sq.w;
    I.hk = I.h / p.group;
    I.delta = I.Lk - I.Lq;
    I.q_tma_row = s0 + kTile * I.t;
    I.o_row = I.q_tma_row;
    I.lse0 = static_cast<int64_t>(I.h) * p.total + s0 + kTile * I.t;
  } else if (!p.bcast) {
    I.Lq = I.Lk;
    I.q_tma_row = s0 + kTile * I.t;
    I.o_row = I.q_tma_row;
    I.lse0 = static_cast<int64_t>(I.h) * p.total + s0 + kTile * I.t;
  } else {
    I.Lq = p.q_len;
    I.q_tma_row = kTile * I.t;
    I.o_row = static_cast<int64_t>(I.b) * p.q_len + kTile * I.t;
    I.lse0 = (static_cast<int64_t>(I.b) * p.heads + I.h) * p.q_len + kTile * I.t;
  }
  I.n_kv = it.w;  // the queue's cost of a forward item is its number of key tiles
  return I;
}

__device__ __forceinline__ FwdStreamItem stream_item(const FwdStreamParams& p, int idx) {
  return item_from(p, p.items[idx], p.item_seq[idx]);
}

// Causal items cost 1 .. n key tiles, very unequal even in longest-first
// order, so they are handed out on demand: the producer warp claims the next
// item with an atomic counter (two items ahead of its loads) and passes each
// record to the other roles through a ring of kRing entries in shared memory;
// an entry with b = -1 ends the stream. A CTA whose items turn out short
// simply claims more, so no CTA idles while another still has items left.
// Non-causal items of one sequence all cost the same and are dealt
// round-robin (CTA c takes c, c + grid, ..), each role reading the records
// itself one item ahead: the ring's hand-offs cost more there than the
// balance gains.
struct ItemRing {
  int4* rec;         // [kRing][2]
  uint64_t* full;    // [kRing], one arrive (the producer)
  uint64_t* empty;   // [kRing], one arrive per consumer warp
};
constexpr int kRingConsumers = 13;  // the MMA warp, eight softmax warps, four epilogue warps

// The order in which the loads are issued (and consumed): Q of an item, then
// K of its first step; for every step j, K of step j + 1 (or the next item's
// Q and first K) before V of step j. claim(I) takes the next item (false at
// the end of the queue); each callback returns false to stop.
template <class FC, class FQ, class FK, class FV>
__device__ __forceinline__ void walk_loads(FC claim, FQ on_q, FK on_k, FV on_v) {
  FwdStreamItem cur, nxt;
  if (!claim(cur)) return;
  bool more = claim(nxt);
  if (!on_q(cur) || !on_k(cur, 0)) return;
  while (true) {
    for (int j = 0; j < cur.n_kv; ++j) {
      if (j + 1 < cur.n_kv) {
        if (!on_k(cur, j + 1)) return;
      } else if (more) {
        if (!on_q(nxt) || !on_k(nxt, 0)) return;
      }
      if (!on_v(cur, j)) return;
    }
    if (!more) return;
    cur = nxt;
    more = claim(nxt);
  }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_stream_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const FwdStreamParams p) {
  using Lay = FwdStreamLayout;
  constexpr int kSlots = Lay::kSlots;
  constexpr int kQS = Lay::kQSlots;
  constexpr uint32_t kIdS = ptx::idesc_bf16(kTile, 128, false, false);  // S = Q K^T
  constexpr uint32_t kIdPV = ptx::idesc_bf16(kTile, kD2, false, true);  // O += P V, P from TMEM

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (smem != smem_raw) {  // base not aligned enough for the layout
    wait_prior_grid();  // the status block was cleared before this kernel
    if (threadIdx.x == 0) atomicCAS(p.status, JFA_OK, JFA_ERR_UNSUPPORTED);
    return;
  }
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
  const ItemRing ring{reinterpret_cast<int4*>(smem + Lay::kOffRing), drain + 3, drain + 3 + Lay::kRing};
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
      ptx::mbar_init(o_free + i, 4);      // the four epilogue warps
      ptx::mbar_init(ml_half + i, kTile);  // every group-0 softmax thread
      ptx::mbar_init(ml_full + i, kTile);  // every group-1 softmax thread
      ptx::mbar_init(ml_empty + i, 4);     // the four epilogue warps
    }
    for (int i = 0; i < 16; ++i) ptx::mbar_init(half_max + i, 1);  // one softmax warp each
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(o_staged, kTile);
    ptx::mbar_init(o_stage_read, 1);
    for (int i = 0; i < Lay::kRing; ++i) {
      ptx::mbar_init(ring.full + i, 1);
      ptx::mbar_init(ring.empty + i, kRingConsumers);
    }
    ctl->abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 12 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
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
  const int n_busy = p.status[3];  // items with at least one key tile: indices 0 .. n_busy - 1
  int32_t* status = p.status;
  const uint64_t budget = p.budget_ns;
  const int cta = blockIdx.x, n_ctas = gridDim.x;
  trace::Writer tw;  // records only in a JFA_TRACE build
  tw.open(status, warp);
  // The next item of a consumer role. Causal: entry k of the item ring (every
  // lane of the warp reads it, lane 0 gives the entry back). Otherwise the
  // role's own round-robin share: st_idx / st_pre hold the next index and its
  // record, read one item ahead. Returns false at the end of the stream or
  // when a wait gave up (ok then turns false as well).
  auto take = [&](uint32_t k, FwdStreamItem& I, bool& ok, int& st_idx, FwdStreamItem& st_pre) -> bool {
    if constexpr (!CAUSAL) {
      (void)k;
      if (st_idx >= n_busy) return false;
      I = st_pre;
      st_idx += n_ctas;
      if (st_idx < n_busy) st_pre = stream_item(p, st_idx);
      return true;
    }
    const uint32_t e = k % Lay::kRing;
    ok = ptx::warp_all(ptx::mbar_wait(ring.full + e, (k / Lay::kRing) & 1, ctl, status, kSiteFwdMmaQ, budget));
    if (!ok) return false;
    const int4 it = ring.rec[2 * e], sq = ring.rec[2 * e + 1];
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ring.empty + e);
    if (it.x < 0) return false;
    I = item_from(p, it, sq);
    return true;
  };

  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t pos = 0, kq = 0;
      auto next_slot = [&](uint32_t& slot) -> bool {
        slot = pos % kSlots;
        const uint32_t round = pos / kSlots;
        if (!ptx::mbar_wait(slot_empty + slot, (round & 1) ^ 1, ctl, status, kSiteFwdProdSlot, budget))
          return false;
        ptx::mbar_arrive_expect_tx(slot_full + slot, Lay::kKVBytes);
        ++pos;
        return true;
      };
      auto on_q = [&](const FwdStreamItem& I) -> bool {
        if (!JFA_TILE_OK(I.t >= 0 && kTile * I.t < I.Lq && I.h >= 0 && I.h < p.heads, ctl, status, kSiteCheckFwdQ))
          return false;
        tw.rec(trace::kFwdStream, trace::kFwdQLoad, kq);
        const uint32_t qs = kq % kQS, qround = kq / kQS;
        if (!ptx::mbar_wait(q_empty + qs, (qround & 1) ^ 1, ctl, status, kSiteFwdProdQ, budget)) return false;
        ptx::mbar_arrive_expect_tx(q_full + qs, Lay::kQBytes);
#pragma unroll
        for (int a = 0; a < 2; ++a)
          ptx::tma_load_2d(smem + Lay::kOffQ + qs * Lay::kQBytes + a * 16384, &tm_q, q_full + qs, I.h * kD2 + 64 * a,
                           I.q_tma_row);
        ++kq;
        return true;
      };
      // K and V tiles: two 64-column atoms of 128 rows each
      auto on_kv = [&](const CUtensorMap* map, const FwdStreamItem& I, int j) -> bool {
        if (!JFA_TILE_OK(j >= 0 && kTile * j < I.Lk && I.hk >= 0, ctl, status, kSiteCheckFwdKV)) return false;
        tw.rec(trace::kFwdStream, trace::kFwdKVLoad, pos);
        uint32_t slot;
        if (!next_slot(slot)) return false;
        uint8_t* dst = smem + Lay::kOffSlots + slot * Lay::kKVBytes;
#pragma unroll
        for (int a = 0; a < 2; ++a)
          ptx::tma_load_2d(dst + a * 16384, map, slot_full + slot, I.hk * kD2 + 64 * a, I.kv_row0 + kTile * j);
        return true;
      };
      uint32_t kc = 0;  // items claimed (ring entries written)
      auto claim = [&](FwdStreamItem& I) -> bool {
        if constexpr (!CAUSAL) {  // round-robin share, read directly
          const int idx = cta + static_cast<int>(kc++) * n_ctas;
          if (idx >= n_busy) return false;
          I = stream_item(p, idx);
          return true;
        }
        const uint32_t e = kc % Lay::kRing;
        if (!ptx::mbar_wait(ring.empty + e, ((kc / Lay::kRing) & 1) ^ 1, ctl, status, kSiteFwdProdQ, budget))
          return false;
        const int idx = atomicAdd(p.counter, 1);
        int4 it = make_int4(-1, 0, 0, 0), sq = make_int4(0, 0, 0, 0);
        if (idx < n_busy) {
          it = p.items[idx];
          sq = p.item_seq[idx];
        }
        ring.rec[2 * e] = it;
        ring.rec[2 * e + 1] = sq;
        ptx::mbar_arrive(ring.full + e);  // release: the record is visible to the entry's waiters
        ++kc;
        if (it.x < 0) return false;
        I = item_from(p, it, sq);
        return true;
      };
      // the walk stops at the first claim past the queue, which wrote the end entry
      // (or at an abort, which the consumers' waits see as well)
      walk_loads(
          claim, on_q, [&](const FwdStreamItem& I, int j) { return on_kv(&tm_k, I, j); },
          [&](const FwdStreamItem& I, int j) { return on_kv(&tm_v, I, j); });
      // After an abort some loads may have no consumer: wait (bounded) for the
      // last fill of every slot so that no copy is in flight when the CTA exits.
      ptx::CtaCtl no_abort{0, 0};
      for (uint32_t i = pos > kSlots ? pos - kSlots : 0; i < pos; ++i)
        ptx::mbar_wait(slot_full + i % kSlots, (i / kSlots) & 1, &no_abort, nullptr, kSiteFwdDrain, budget);
      for (uint32_t i = kq > kQS ? kq - kQS : 0; i < kq; ++i)
        ptx::mbar_wait(q_full + i % kQS, (i / kQS) & 1, &no_abort, nullptr, kSiteFwdDrain, budget);
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (so every value it computes is warp-uniform)
    // and one elected lane issues each group of MMAs and commits.
    uint32_t pos = 0;
    bool ok = true;
    auto slot_wait = [&](uint32_t& slot) -> bool {
      slot = pos % kSlots;
      const uint32_t round = pos / kSlots;
      const bool w = ptx::mbar_wait(slot_full + slot, round & 1, ctl, status, kSiteFwdMmaSlot, budget);
      ptx::tc_fence_after();
      ++pos;
      return ptx::warp_all(w);
    };
    auto q_wait = [&](uint32_t kq) -> bool {
      const uint32_t qs = kq % kQS, qround = kq / kQS;
      const bool w = ptx::mbar_wait(q_full + qs, qround & 1, ctl, status, kSiteFwdMmaQ, budget);
      ptx::tc_fence_after();
      return ptx::warp_all(w);
    };
    // S(x) = Q K^T into S buffer x & 1. Descriptors are built once per tile; a
    // K step adds its byte offset / 16 to the start-address field (no carry:
    // shared addresses are < 2^18). last_q_use releases the Q buffer.
    auto issue_s = [&](uint32_t kq, uint32_t x, bool last_q_use) -> bool {
      uint32_t slot;
      if (!slot_wait(slot)) return false;
      const uint32_t qs = kq % kQS;
      const uint64_t q_desc = ptx::sdesc_sw128(ptx::smem_u32(smem + Lay::kOffQ + qs * Lay::kQBytes), 16, 1024);
      const uint64_t k_desc =
          ptx::sdesc_sw128(ptx::smem_u32(smem + Lay::kOffSlots + slot * Lay::kKVBytes), 16, 1024);
      const uint32_t d_tmem = tmem + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
      if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdSIssue, x);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kD2 / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          ptx::mma_ss(d_tmem, q_desc + (off >> 4), k_desc + (off >> 4), kIdS, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(s_full + (x & 1));
        ptx::mma_commit(slot_empty + slot);
        if (last_q_use) ptx::mma_commit(q_empty + qs);
      }
      __syncwarp();
      return true;
    };
    FwdStreamItem cur, nxt, st_pre;
    int st_idx = cta;  // round-robin share (non-causal)
    if (!CAUSAL && st_idx < n_busy) st_pre = stream_item(p, st_idx);
    uint32_t kr = 0;  // ring entries taken
    bool have = take(kr++, cur, ok, st_idx, st_pre);
    uint32_t kq = 0, x = 0;  // busy items so far, steps so far
    if (have) ok = q_wait(0) && issue_s(0, 0, cur.n_kv == 1);
    while (ok && have) {
      const bool more = take(kr++, nxt, ok, st_idx, st_pre);
      if (!ok) break;
      const int n = cur.n_kv;
      const uint32_t ob = kq & 1;
      for (int j = 0; ok && j < n; ++j, ++x) {
        if (j + 1 < n) {
          if (!(ok = issue_s(kq, x + 1, j + 2 == n))) break;
        } else if (more) {
          if (!(ok = q_wait(kq + 1) && issue_s(kq + 1, x + 1, nxt.n_kv == 1))) break;
        }
        // V of this step (loaded long before) and the O buffer first, so that
        // PV issues as soon as P is ready
        uint32_t slot;
        if (!(ok = slot_wait(slot))) break;
        bool w = true;
        if (j == 0 && kq >= 2)  // the epilogue of item kq - 2 has read this O buffer
          w = ptx::mbar_wait(o_free + ob, ((kq - 2) >> 1) & 1, ctl, status, kSiteFwdMmaOFree, budget);
        w = w && ptx::mbar_wait(p_full + (x & 1), (x >> 1) & 1, ctl, status, kSiteFwdMmaP, budget);
        if (!(ok = ptx::warp_all(w))) break;
        ptx::tc_fence_after();
        const uint64_t v_desc =
            ptx::sdesc_sw128(ptx::smem_u32(smem + Lay::kOffSlots + slot * Lay::kKVBytes), 16384, 1024);
        const uint32_t p_tmem = tmem + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
        const uint32_t o_tmem = tmem + (ob ? Lay::kColO1 : Lay::kColO0);
        if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdPVIssue, x);
        if (ptx::elect_one()) {
          // keys 16 kk ..: group 0's P (keys 0-63) at S columns 0-31, group 1's
          // (keys 64-127) at S columns 64-95
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            ptx::mma_ts(o_tmem, p_tmem + (kk >> 2) * 64 + (kk & 3) * 8, v_desc + ((kk * 2048) >> 4), kIdPV,
                        (j > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(o_ready + (x & 1));
          ptx::mma_commit(slot_empty + slot);
          if (j + 1 == n) ptx::mma_commit(o_final + ob);
        }
        __syncwarp();
      }
      ++kq;
      cur = nxt;
      have = more;
    }
    if (ptx::elect_one()) ptx::mma_commit(drain);
    __syncwarp();
    ptx::CtaCtl no_abort{0, 0};
    ptx::mbar_wait(drain, 0, &no_abort, nullptr, kSiteFwdDrain, budget);
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int g = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int c_own = 64 * g, c_other = 64 - c_own;  // first key column of this group's / the other group's half
    const float sl = p.scale_log2;
    uint32_t x = 0, kq = 0;
    bool ok = true, s_ready = false;  // s_ready: S of step x is known to be complete
    uint32_t kr = 0;  // ring entries taken
    FwdStreamItem I, st_pre;
    int st_idx = cta;  // round-robin share (non-causal)
    if (!CAUSAL && st_idx < n_busy) st_pre = stream_item(p, st_idx);
    while (ok && take(kr++, I, ok, st_idx, st_pre)) {
      const int n = I.n_kv;
      const uint32_t ob = kq & 1;
      const uint32_t o_tmem = tmem + lane_base + (ob ? Lay::kColO1 : Lay::kColO0) + c_own;
      const int qi = kTile * I.t + r;  // query position in its sequence
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j, ++x) {
        const uint32_t s_tmem = tmem + lane_base + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
        if (!s_ready && !(ok = ptx::mbar_wait(s_full + (x & 1), (x >> 1) & 1, ctl, status, kSiteFwdSoftS, budget)))
          break;
        ptx::tc_fence_after();
        if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdSoftBegin, x);
        // keys j*128 + c with c >= lim are masked (past the sequence, or past
        // the bottom-right aligned diagonal: key j visible iff j <= qi + delta)
        const int lim = CAUSAL ? min(qi + 1 + I.delta - kTile * j, I.Lk - kTile * j) : I.Lk - kTile * j;
        auto mask = [&](uint32_t(&v)[32], int c0) {
          if (lim < c0 + 32) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c0 + e >= lim) v[e] = __float_as_uint(-INFINITY);
          }
        };
        // this group's half of the row (it stays in registers) and its maximum,
        // folded in eight independent chains of three-input maxima
        uint32_t sa[2][32];
        ptx::tmem_ld32(s_tmem + c_own, sa[0]);
        ptx::tmem_ld32(s_tmem + c_own + 32, sa[1]);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(sa[0]);
        ptx::reg_fence32(sa[1]);
        mask(sa[0], c_own);
        mask(sa[1], c_own + 32);
        if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdSoftLoaded, x);
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
        // The two groups exchange their halves' maxima (neither reads the
        // other's scores): each writes its maximum into the last column of its
        // own half of S, which it no longer needs (P goes over the first 32).
        // After the first step of an item the exponentials are taken against
        // the running max at once, and taken again only if the row max turns
        // out to have grown by more than 2^8 (both groups see the same two
        // maxima, so they decide alike).
        tmem_st1(s_tmem + c_own + 63, __float_as_uint(hmax));
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(half_max + ((x & 1) * 2 + g) * 4 + quarter);
        if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdSoftPub, x);
        uint64_t* other = half_max + ((x & 1) * 2 + (1 - g)) * 4 + quarter;
        auto other_max = [&]() -> float {  // after `other` has completed
          ptx::tc_fence_after();
          const uint32_t v = tmem_ld1(s_tmem + c_other + 63);
          ptx::tmem_ld_wait();
          return __uint_as_float(v);
        };
        // P = 2^(S sl - m) over this group's half, stored over its S columns; returns the half-row sum
        const uint64_t sl2 = ptx::f2_packf(sl, sl);
        auto exps = [&](float mref) -> float {
          const float mu = (mref == -INFINITY) ? 0.f : mref;  // a row with no visible key yet keeps P = 0
          const uint64_t nmu2 = ptx::f2_packf(-mu, -mu);
          uint64_t ls2[2] = {ptx::f2_packf(0.f, 0.f), ptx::f2_packf(0.f, 0.f)};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x0, x1;
              ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(sa[u][2 * e], sa[u][2 * e + 1]), sl2, nmu2), x0, x1);
              const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
              ls2[e & 1] = ptx::f2_add(ls2[e & 1], ptx::f2_packf(p0, p1));
              pk[e] = ptx::pack_bf16(p0, p1);
            }
            ptx::tmem_st16(s_tmem + c_own + 16 * u, pk);
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
          if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdSoftMax, x);
          lsum = exps(m);
          if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdSoftExp, x);
        } else {
          lsum = exps(m);
          if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdSoftExp, x);
          if (!(ok = ptx::mbar_wait(other, (x >> 1) & 1, ctl, status, kSiteFwdSoftS, budget))) break;
          const float mnew = fmaxf(hmax, other_max()) * sl;
          if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdSoftMax, x);
          // O is rescaled only when the running max grows by more than 2^8;
          // otherwise the old max stays the reference and P stays below 2^8.
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
            l *= f;
            m = mm;
            lsum = exps(m);  // again, against the new reference (over the first try's P)
          }
        }
        l += lsum;
        if (j + 1 == n) {
          // Row statistics of the finished item go to the epilogue: group 0
          // stores (m, its sum), group 1 adds its sum to that.
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
        // S of the next step (usually long complete), tested while the P stores drain
        s_ready = ptx::mbar_test(s_full + ((x + 1) & 1), ((x + 1) >> 1) & 1);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full + (x & 1));
        if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdSoftEnd, x);
      }
      ++kq;
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 8-11)
    // O of a whole query tile leaves by TMA store: normalised, packed to bf16
    // and staged (128B swizzle, two 64-column atoms); a partial tile, whose
    // 128-row box would reach into the next sequence, is stored row by row.
    const int quarter = warp & 3;  // TMEM lanes 32 (warp % 4) .. are this warp's rows
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr float kLn2 = 0.6931471805599453f;
    const bool issuer = warp == 8 && lane == 0;
    uint8_t* ostage = smem + Lay::kOffOStage;
    uint32_t kq = 0, n_st = 0;  // busy items; items whose O went through the staging
    // items with no key (they follow the busy ones): O = 0, LSE = -inf, dealt statically
    for (int idx = n_busy + cta; idx < n_items; idx += n_ctas) {
      const FwdStreamItem I = stream_item(p, idx);
      const int qi = kTile * I.t + r;
      __nv_bfloat16* orow = p.o + (I.o_row + r) * static_cast<int64_t>(p.heads) * kD2 + static_cast<int64_t>(I.h) * kD2;
      if (qi < I.Lq) {
        for (int c = 0; c < kD2; c += 8) ptx::st_v4(orow + c, 0, 0, 0, 0);
        p.lse[I.lse0 + r] = -INFINITY;
      }
    }
    uint32_t kr = 0;  // ring entries taken
    bool ok = true;
    FwdStreamItem I, st_pre;
    int st_idx = cta;  // round-robin share (non-causal)
    if (!CAUSAL && st_idx < n_busy) st_pre = stream_item(p, st_idx);
    while (ok && take(kr++, I, ok, st_idx, st_pre)) {
      const int qi = kTile * I.t + r;
      const bool row_ok = qi < I.Lq;
      __nv_bfloat16* orow = p.o + (I.o_row + r) * static_cast<int64_t>(p.heads) * kD2 + static_cast<int64_t>(I.h) * kD2;
      const uint32_t ob = kq & 1;
      bool w = ptx::mbar_wait(o_final + ob, (kq >> 1) & 1, ctl, status, kSiteFwdEpi, budget);
      w = w && ptx::mbar_wait(ml_full + ob, (kq >> 1) & 1, ctl, status, kSiteFwdEpi, budget);
      if (!w) break;
      ptx::tc_fence_after();
      if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdEpiBegin, kq);
      const float2 st = ml[ob * kTile + r];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ml_empty + ob);
      const float inv_l = st.y > 0.f ? 1.0f / st.y : 0.f;
      const uint32_t o_tmem = tmem + lane_base + (ob ? Lay::kColO1 : Lay::kColO0);
      const bool staged = I.Lq - kTile * I.t >= kTile;
      if (staged && n_st > 0) {  // the previous TMA store has read the staging
        if (issuer) {
          ptx::bulk_wait_read0();
          ptx::mbar_arrive(o_stage_read);
        }
        if (!ptx::mbar_wait(o_stage_read, (n_st - 1) & 1, ctl, status, kSiteFwdEpi, budget)) break;
      }
#pragma unroll 1
      for (int c = 0; c < kD2 / 32; ++c) {
        uint32_t ov[32];
        ptx::tmem_ld32(o_tmem + 32 * c, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(ov);
        if (c == kD2 / 32 - 1) {  // all of O is in registers: the next item may use this buffer
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(o_free + ob);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            wv[e] = ptx::pack_bf16(__uint_as_float(ov[8 * q4 + 2 * e]) * inv_l,
                                   __uint_as_float(ov[8 * q4 + 2 * e + 1]) * inv_l);
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
          ptx::tma_store_2d(&tm_o, ostage, I.h * kD2, static_cast<int32_t>(I.o_row));
          ptx::tma_store_2d(&tm_o, ostage + 16384, I.h * kD2 + 64, static_cast<int32_t>(I.o_row));
          ptx::bulk_commit();
        }
        ++n_st;
      }
      if (row_ok) p.lse[I.lse0 + r] = (st.x + log2f(st.y)) * kLn2;
      if (lane == 0) tw.rec(trace::kFwdStream, trace::kFwdEpiEnd, kq);
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

template <bool CAUSAL>
cudaError_t launch_fwd_stream_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, const FwdStreamParams& p, int grid, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(fwd_stream_kernel<CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FwdStreamLayout::kBytes);
  });
  if (e != cudaSuccess) return e;
  return launch_after(fwd_stream_kernel<CAUSAL>, dim3(grid), dim3(kThreads), FwdStreamLayout::kBytes, stream, tq, tk, tv,
                      to, p);
}

}  // namespace

cudaError_t launch_fwd_stream(bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, const int4* items, const int4* item_seq, const VarInfo& var,
                              int32_t* status, void* o, float* lse, int heads, int total, int bcast, int q_len,
                              float scale, uint64_t budget_ns, int grid, cudaStream_t stream) {
  FwdStreamParams p;
  p.items = items;
  p.item_seq = item_seq;
  p.status = status;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.heads = heads;
  p.total = total;
  p.bcast = bcast;
  p.q_len = q_len;
  p.var = var.var;
  p.group = var.group;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.budget_ns = budget_ns;
  p.counter = status + kStatusItemCounter;
  return causal ? launch_fwd_stream_t<true>(tq, tk, tv, to, p, grid, stream)
                : launch_fwd_stream_t<false>(tq, tk, tv, to, p, grid, stream);
}

}  // namespace jfa
