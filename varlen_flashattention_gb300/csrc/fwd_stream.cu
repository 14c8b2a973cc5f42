// Jagged FlashAttention forward as a flat stream of steps, head_dim 128, on
// CTA pairs (tcgen05 cta_group::2) or on single CTAs.
//
// What it computes is the forward of fwd.cu ("Cutting-edge isn't
// plug-and-play: customizing FA4 on B300", FlashAttention recap; "Optimizing
// Jagged Flash Attention with TLX", third paragraph). The difference is how
// the tensor cores are driven ("Optimizing Jagged Flash Attention with TLX",
// fifth paragraph: the 2-CTA collaborative MMA adopted from FA4): two CTAs on
// two SMs form a cluster and work on two query tiles of the same sequence and
// head. Every MMA has M = 256 (CTA r holds rows 128r..128r+127 of Q, S, P, O
// in its own shared memory / TMEM) and the B operand is split along N: CTA r
// loads key rows 64r..64r+63 of each K tile and head-dim columns 64r..64r+63
// of each V tile, so each SM reads half of every K/V tile from L2 and from
// its shared memory.
//
// The work of a cluster is one flat stream of steps (one step = one key/value
// tile of one item), so that nothing drains between items: the S = Q K^T of
// the next step is issued before the P V of the current one even when the next
// step belongs to the next item, O is double-buffered in TMEM (items alternate
// between the two accumulators), and separate epilogue warps normalise and
// store an item's O while the next item is computed.
//
// The single-CTA form (PAIR = false) is the same pipeline with M = 128 MMAs,
// whole K/V tiles in every CTA and no cross-SM signals.
//
// Roles (both CTAs, 320 threads): warps 0-3 softmax (thread = query row =
// TMEM lane), warps 4-7 epilogue, warp 8 TMA producer. Warp 9 of CTA 0 issues
// every MMA (the whole warp runs the loop, one elected lane issues); its
// commits arrive on the same barrier in both CTAs. Warp 9 of CTA 1 forwards
// the completion of its own TMA loads to CTA 0 (remote mbarrier arrive), and
// CTA 1's softmax and epilogue warps signal "P ready" and "O free" to CTA 0
// the same way. With ten warps a thread has at most 168 registers, so the
// softmax keeps half of a score row in registers and reads the other half
// from TMEM twice.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "jfa_internal.h"
#include "ptx.cuh"

namespace jfa {

namespace {

constexpr int kD2 = 128;

struct FwdStreamParams {
  const int32_t* offsets;
  const int4* items;  // (b, h, pair u, cost)
  int32_t* status;
  __nv_bfloat16* o;
  float* lse;
  int32_t heads, total, bcast, q_len;
  float scale_log2;
  uint64_t budget_ns;
};

template <bool PAIR>
struct FwdStreamLayout {
  static constexpr int kQBytes = kTile * kD2 * 2;  // own query tile: 128 rows x 128 d
  // a slot holds half a K tile (64 rows) or half a V tile (64 columns) on a
  // pair, a whole K or V tile on a single CTA
  static constexpr int kHalfBytes = PAIR ? 16384 : 32768;
  static constexpr int kQSlots = 2;
  static constexpr int kSlots = PAIR ? 9 : 5;
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = kQSlots * kQBytes;
  static constexpr int kOffMl = kOffSlots + kSlots * kHalfBytes;  // float2 (m, l) per row, two buffers
  static constexpr int kOffBars = kOffMl + 2 * kTile * 8;
  // q_full[2], q_peer[2], q_empty[2], slot_full[S], slot_peer[S], slot_empty[S],
  // s_full[2], p_full[2], o_ready[2], o_final[2], o_free[2], ml_full[2], ml_empty[2], drain
  static constexpr int kNumBars = 3 * kQSlots + 3 * kSlots + 7 * 2 + 1;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64;
  // Tiles need 1024-byte alignment; the dynamic shared-memory base is 1024-byte
  // aligned on this part (a kernel that finds it otherwise reports
  // JFA_ERR_UNSUPPORTED), so no slack is reserved on a single CTA.
  static constexpr int kAlloc = kBytes + (PAIR ? 1024 : 0);
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384, kTmemCols = 512;
  static_assert(kAlloc <= 232448, "shared memory budget");
};

struct FwdStreamItem {
  int b, h, u, t;  // t = this CTA's query tile (2u + rank)
  int q_tma_row, kv_row0, Lq, Lk, n_kv;
  int64_t o_row, lse0;
};

template <bool CAUSAL, bool PAIR>
__device__ __forceinline__ FwdStreamItem stream_item(const FwdStreamParams& p, int idx, uint32_t rank) {
  const int4 it = p.items[idx];
  FwdStreamItem I;
  I.b = it.x;
  I.h = it.y;
  I.u = it.z;
  I.t = PAIR ? 2 * I.u + static_cast<int>(rank) : I.u;
  const int s0 = p.offsets[I.b], s1 = p.offsets[I.b + 1];
  I.Lk = s1 - s0;
  I.kv_row0 = s0;
  if (!p.bcast) {
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
  const int nk = (I.Lk + kTile - 1) / kTile;
  // the same for both CTAs of a pair
  I.n_kv = CAUSAL ? min(PAIR ? 2 * I.u + 2 : I.u + 1, nk) : nk;
  return I;
}

// The next item of this cluster with at least one key/value tile, starting at
// index idx. Returns its index (>= n_items when there is none).
template <bool CAUSAL, bool PAIR>
__device__ __forceinline__ int next_busy(const FwdStreamParams& p, int idx, int stride, int n_items, uint32_t rank,
                                         FwdStreamItem& I) {
  for (; idx < n_items; idx += stride) {
    I = stream_item<CAUSAL, PAIR>(p, idx, rank);
    if (I.n_kv > 0) break;
  }
  return idx;
}

// The order in which a CTA's loads are issued (and consumed): Q of an item,
// then K of its first step; for every step j, K of step j + 1 (or the next
// item's Q and first K) before V of step j. The producer and the forwarder of
// CTA 1 both walk it. Each callback returns false to stop the walk.
template <bool CAUSAL, bool PAIR, class FQ, class FK, class FV>
__device__ __forceinline__ void walk_loads(const FwdStreamParams& p, uint32_t rank, int first, int stride, int n_items,
                                           FQ on_q, FK on_k, FV on_v) {
  FwdStreamItem cur, nxt;
  int idx = next_busy<CAUSAL, PAIR>(p, first, stride, n_items, rank, cur);
  if (idx >= n_items) return;
  if (!on_q(cur) || !on_k(cur, 0)) return;
  while (true) {
    const int nidx = next_busy<CAUSAL, PAIR>(p, idx + stride, stride, n_items, rank, nxt);
    const bool more = nidx < n_items;
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
    idx = nidx;
  }
}

// Launched with a cluster of 2 (PAIR) or 1. tm_k reads 64-row boxes on a pair
// (each CTA loads half of a key tile) and 128-row boxes on a single CTA.
template <bool CAUSAL, bool PAIR>
__global__ void __launch_bounds__(320, 1)
    fwd_stream_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdStreamParams p) {
  using Lay = FwdStreamLayout<PAIR>;
  constexpr int kM = PAIR ? 256 : 128;
  constexpr int kKAtom = PAIR ? 8192 : 16384;  // bytes of one 64-column atom of the K rows a CTA holds
  constexpr uint32_t kPeers = PAIR ? 8 : 4;   // softmax / epilogue warps that signal the issuing CTA
  constexpr int kSlots = Lay::kSlots;
  constexpr int kQS = Lay::kQSlots;
  constexpr uint32_t kIdS = ptx::idesc_bf16(kM, 128, false, false);  // S = Q K^T (M = 256 over a pair)
  constexpr uint32_t kIdPV = ptx::idesc_bf16(kM, kD2, false, true);  // O += P V, P from TMEM

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (smem + Lay::kBytes > smem_raw + Lay::kAlloc) {  // base not aligned enough for the layout
    if (threadIdx.x == 0) atomicCAS(p.status, JFA_OK, JFA_ERR_UNSUPPORTED);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBars);
  uint64_t* q_full = bars;
  uint64_t* q_peer = q_full + kQS;
  uint64_t* q_empty = q_peer + kQS;
  uint64_t* slot_full = q_empty + kQS;
  uint64_t* slot_peer = slot_full + kSlots;
  uint64_t* slot_empty = slot_peer + kSlots;
  uint64_t* s_full = slot_empty + kSlots;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_ready = p_full + 2;
  uint64_t* o_final = o_ready + 2;
  uint64_t* o_free = o_final + 2;
  uint64_t* ml_full = o_free + 2;
  uint64_t* ml_empty = ml_full + 2;
  uint64_t* drain = ml_empty + 2;
  float2* ml = reinterpret_cast<float2*>(smem + Lay::kOffMl);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  ptx::CtaCtl* ctl = reinterpret_cast<ptx::CtaCtl*>(smem + Lay::kOffMisc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? ptx::cluster_rank() : 0;
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQS; ++i) {
      ptx::mbar_init(q_full + i, 1);
      ptx::mbar_init(q_peer + i, 1);
      ptx::mbar_init(q_empty + i, 1);
    }
    for (int i = 0; i < kSlots; ++i) {
      ptx::mbar_init(slot_full + i, 1);
      ptx::mbar_init(slot_peer + i, 1);
      ptx::mbar_init(slot_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(s_full + i, 1);
      ptx::mbar_init(p_full + i, kPeers);  // four softmax warps in each CTA
      ptx::mbar_init(o_ready + i, 1);
      ptx::mbar_init(o_final + i, 1);
      ptx::mbar_init(o_free + i, kPeers);  // four epilogue warps in each CTA
      ptx::mbar_init(ml_full + i, kTile);  // every softmax thread of this CTA
      ptx::mbar_init(ml_empty + i, 4);     // the four epilogue warps of this CTA
    }
    ptx::mbar_init(drain, 1);
    ctl->abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
  }
  __syncthreads();
  if (PAIR) ptx::cluster_sync();  // barriers of both CTAs initialised before any remote arrive
  if (warp == 9) {
    if (PAIR) {
      ptx::tmem_alloc2(tmem_slot, Lay::kTmemCols);  // both CTAs of the pair allocate together
      ptx::tmem_relinquish2();
    } else {
      ptx::tmem_alloc(tmem_slot, Lay::kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();  // TMEM allocated in both CTAs before the first MMA
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_items = p.status[2];
  int32_t* status = p.status;
  const uint64_t budget = p.budget_ns;
  const int cluster = PAIR ? blockIdx.x >> 1 : blockIdx.x, n_clusters = PAIR ? gridDim.x >> 1 : gridDim.x;
  // waits on barriers that the other CTA of a pair arrives on (cluster scope)
  auto wait_x = [&](uint64_t* bar, uint32_t parity, ptx::CtaCtl* c, int32_t* st, int where, uint64_t b) -> bool {
    return PAIR ? ptx::mbar_wait_cluster(bar, parity, c, st, where, b) : ptx::mbar_wait(bar, parity, c, st, where, b);
  };
  auto commit = [&](uint64_t* bar) {  // arrives on bar in every CTA of the pair
    if (PAIR)
      ptx::mma2_commit(bar, 0x3);
    else
      ptx::mma_commit(bar);
  };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t pos = 0, kq = 0;
      auto next_slot = [&](uint32_t& slot) -> bool {
        slot = pos % kSlots;
        const uint32_t round = pos / kSlots;
        if (!wait_x(slot_empty + slot, (round & 1) ^ 1, ctl, status, kSiteFwdProdSlot, budget))
          return false;
        ptx::mbar_arrive_expect_tx(slot_full + slot, Lay::kHalfBytes);
        ++pos;
        return true;
      };
      auto on_q = [&](const FwdStreamItem& I) -> bool {
        const uint32_t qs = kq % kQS, qround = kq / kQS;
        if (!wait_x(q_empty + qs, (qround & 1) ^ 1, ctl, status, kSiteFwdProdQ, budget)) return false;
        ptx::mbar_arrive_expect_tx(q_full + qs, Lay::kQBytes);
#pragma unroll
        for (int a = 0; a < 2; ++a)
          ptx::tma_load_2d(smem + Lay::kOffQ + qs * Lay::kQBytes + a * 16384, &tm_q, q_full + qs, I.h * kD2 + 64 * a,
                           I.q_tma_row);
        ++kq;
        return true;
      };
      // pair: key rows 64 rank .. of tile j, all of d; single: the whole tile
      auto on_k = [&](const FwdStreamItem& I, int j) -> bool {
        uint32_t slot;
        if (!next_slot(slot)) return false;
        uint8_t* dst = smem + Lay::kOffSlots + slot * Lay::kHalfBytes;
#pragma unroll
        for (int a = 0; a < 2; ++a)
          ptx::tma_load_2d(dst + a * kKAtom, &tm_k, slot_full + slot, I.h * kD2 + 64 * a,
                           I.kv_row0 + kTile * j + 64 * static_cast<int>(rank));
        return true;
      };
      // pair: all key rows of tile j, head-dim columns 64 rank ..; single: the whole tile
      auto on_v = [&](const FwdStreamItem& I, int j) -> bool {
        uint32_t slot;
        if (!next_slot(slot)) return false;
#pragma unroll
        for (int a = 0; a < (PAIR ? 1 : 2); ++a)
          ptx::tma_load_2d(smem + Lay::kOffSlots + slot * Lay::kHalfBytes + a * 16384, &tm_v, slot_full + slot,
                           I.h * kD2 + 64 * (static_cast<int>(rank) + a), I.kv_row0 + kTile * j);
        return true;
      };
      walk_loads<CAUSAL, PAIR>(p, rank, cluster, n_clusters, n_items, on_q, on_k, on_v);
      // After an abort some loads may have no consumer: wait (bounded) for the
      // last fill of every slot so that no copy is in flight when the CTA exits.
      ptx::CtaCtl no_abort{0, 0};
      for (uint32_t i = pos > kSlots ? pos - kSlots : 0; i < pos; ++i)
        ptx::mbar_wait(slot_full + i % kSlots, (i / kSlots) & 1, &no_abort, nullptr, kSiteFwdDrain, budget);
      for (uint32_t i = kq > kQS ? kq - kQS : 0; i < kq; ++i)
        ptx::mbar_wait(q_full + i % kQS, (i / kQS) & 1, &no_abort, nullptr, kSiteFwdDrain, budget);
    }
  } else if (warp == 9 && leader) {
    // ------------------------------------------------------------ MMA issuer (CTA 0)
    // The whole warp runs the loop (so every value it computes is warp-uniform)
    // and one elected lane issues each group of MMAs and commits.
    uint32_t pos = 0;
    bool ok = true;
    auto slot_wait = [&](uint32_t& slot) -> bool {
      slot = pos % kSlots;
      const uint32_t round = pos / kSlots;
      bool w = ptx::mbar_wait(slot_full + slot, round & 1, ctl, status, kSiteFwdMmaSlot, budget);
      if (PAIR) w = w && wait_x(slot_peer + slot, round & 1, ctl, status, kSiteFwdMmaSlot, budget);
      ptx::tc_fence_after();
      ++pos;
      return ptx::warp_all(w);
    };
    auto q_wait = [&](uint32_t kq) -> bool {
      const uint32_t qs = kq % kQS, qround = kq / kQS;
      bool w = ptx::mbar_wait(q_full + qs, qround & 1, ctl, status, kSiteFwdMmaQ, budget);
      if (PAIR) w = w && wait_x(q_peer + qs, qround & 1, ctl, status, kSiteFwdMmaQ, budget);
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
          ptx::sdesc_sw128(ptx::smem_u32(smem + Lay::kOffSlots + slot * Lay::kHalfBytes), 16, 1024);
      const uint32_t d_tmem = tmem + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
      if (ptx::elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kD2 / 16; ++kk) {
          const uint32_t qo = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t ko = (kk >> 2) * kKAtom + (kk & 3) * 32;
          if (PAIR)
            ptx::mma2_ss(d_tmem, q_desc + (qo >> 4), k_desc + (ko >> 4), kIdS, kk > 0 ? 1u : 0u);
          else
            ptx::mma_ss(d_tmem, q_desc + (qo >> 4), k_desc + (ko >> 4), kIdS, kk > 0 ? 1u : 0u);
        }
        commit(s_full + (x & 1));
        commit(slot_empty + slot);
        if (last_q_use) commit(q_empty + qs);
      }
      __syncwarp();
      return true;
    };
    FwdStreamItem cur, nxt;
    int idx = next_busy<CAUSAL, PAIR>(p, cluster, n_clusters, n_items, rank, cur);
    uint32_t kq = 0, x = 0;  // busy items so far, steps so far
    if (idx < n_items) ok = q_wait(0) && issue_s(0, 0, cur.n_kv == 1);
    while (ok && idx < n_items) {
      const int nidx = next_busy<CAUSAL, PAIR>(p, idx + n_clusters, n_clusters, n_items, rank, nxt);
      const bool more = nidx < n_items;
      const int n = cur.n_kv;
      const uint32_t ob = kq & 1;
      for (int j = 0; ok && j < n; ++j, ++x) {
        if (j + 1 < n) {
          if (!(ok = issue_s(kq, x + 1, j + 2 == n))) break;
        } else if (more) {
          if (!(ok = q_wait(kq + 1) && issue_s(kq + 1, x + 1, nxt.n_kv == 1))) break;
        }
        bool w = wait_x(p_full + (x & 1), (x >> 1) & 1, ctl, status, kSiteFwdMmaP, budget);
        if (j == 0 && kq >= 2)  // the epilogue of item kq - 2 has read this O buffer
          w = w && wait_x(o_free + ob, ((kq - 2) >> 1) & 1, ctl, status, kSiteFwdMmaOFree, budget);
        if (!(ok = ptx::warp_all(w))) break;
        uint32_t slot;
        if (!(ok = slot_wait(slot))) break;
        const uint64_t v_desc =
            ptx::sdesc_sw128(ptx::smem_u32(smem + Lay::kOffSlots + slot * Lay::kHalfBytes), 16384, 1024);
        const uint32_t p_tmem = tmem + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
        const uint32_t o_tmem = tmem + (ob ? Lay::kColO1 : Lay::kColO0);
        if (ptx::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            if (PAIR)
              ptx::mma2_ts(o_tmem, p_tmem + kk * 8, v_desc + ((kk * 2048) >> 4), kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
            else
              ptx::mma_ts(o_tmem, p_tmem + kk * 8, v_desc + ((kk * 2048) >> 4), kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
          }
          commit(o_ready + (x & 1));
          commit(slot_empty + slot);
          if (j + 1 == n) commit(o_final + ob);
        }
        __syncwarp();
      }
      ++kq;
      cur = nxt;
      idx = nidx;
    }
    if (ptx::elect_one()) {
      if (PAIR)
        ptx::mma2_commit(drain, 0x1);
      else
        ptx::mma_commit(drain);
    }
    __syncwarp();
    ptx::CtaCtl no_abort{0, 0};
    ptx::mbar_wait(drain, 0, &no_abort, nullptr, kSiteFwdDrain, budget);
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ load forwarder (CTA 1 of a pair)
    // Tells CTA 0 that this CTA's halves of Q and of every K/V tile have landed.
    if (lane == 0) {
      uint32_t pos = 0, kq = 0;
      auto on_q = [&](const FwdStreamItem&) -> bool {
        const uint32_t qs = kq % kQS, qround = kq / kQS;
        if (!ptx::mbar_wait(q_full + qs, qround & 1, ctl, status, kSiteFwdMmaQ, budget)) return false;
        ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(q_peer + qs), 0));
        ++kq;
        return true;
      };
      auto on_slot = [&](const FwdStreamItem&, int) -> bool {
        const uint32_t slot = pos % kSlots, round = pos / kSlots;
        if (!ptx::mbar_wait(slot_full + slot, round & 1, ctl, status, kSiteFwdMmaSlot, budget)) return false;
        ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(slot_peer + slot), 0));
        ++pos;
        return true;
      };
      walk_loads<CAUSAL, PAIR>(p, rank, cluster, n_clusters, n_items, on_q, on_slot, on_slot);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax (warps 0-3, both CTAs)
    const int r = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float sl = p.scale_log2;
    // "P ready" goes to CTA 0's barrier: locally in CTA 0, remotely from CTA 1
    auto signal_p = [&](uint64_t* bar) {
      if (lane != 0) return;
      if (!PAIR || leader)
        ptx::mbar_arrive(bar);
      else
        ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(bar), 0));
    };
    uint32_t x = 0, kq = 0;
    bool ok = true;
    for (int idx = cluster; ok && idx < n_items; idx += n_clusters) {
      const FwdStreamItem I = stream_item<CAUSAL, PAIR>(p, idx, rank);
      const int n = I.n_kv;
      if (n == 0) continue;
      const uint32_t ob = kq & 1;
      const uint32_t o_tmem = tmem + lane_base + (ob ? Lay::kColO1 : Lay::kColO0);
      const int qi = kTile * I.t + r;  // query position in its sequence
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j, ++x) {
        const uint32_t s_tmem = tmem + lane_base + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
        if (!(ok = wait_x(s_full + (x & 1), (x >> 1) & 1, ctl, status, kSiteFwdSoftS, budget))) break;
        ptx::tc_fence_after();
        // Columns 0-63 of S are overwritten by P (bf16 pairs), so score chunks 0
        // and 1 stay in registers; chunks 2 and 3 are read again for the exps.
        uint32_t sa[2][32], sb[32];
        ptx::tmem_ld32(s_tmem, sa[0]);
        ptx::tmem_ld32(s_tmem + 32, sa[1]);
        ptx::tmem_ld32(s_tmem + 64, sb);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(sa[0]);
        ptx::reg_fence32(sa[1]);
        ptx::reg_fence32(sb);
        // keys j*128 + c with c >= lim are masked (past the sequence, or above the diagonal)
        const int lim = CAUSAL ? min(qi + 1 - kTile * j, I.Lk - kTile * j) : I.Lk - kTile * j;
        auto mask = [&](uint32_t(&v)[32], int c0) {
          if (lim < c0 + 32) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c0 + e >= lim) v[e] = __float_as_uint(-INFINITY);
          }
        };
        mask(sa[0], 0);
        mask(sa[1], 32);
        mask(sb, 64);
        // row max: eight independent chains of three-input maxima
        float mx8[8];
        auto fold = [&](const uint32_t(&v)[32], int e0) {
#pragma unroll
          for (int e = e0; e < 32; e += 2)
            mx8[(e >> 1) & 7] = ptx::fmax3(mx8[(e >> 1) & 7], __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
        };
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(__uint_as_float(sa[0][2 * k]), __uint_as_float(sa[0][2 * k + 1]));
        fold(sa[0], 16);
        fold(sa[1], 0);
        fold(sb, 0);
        ptx::tmem_ld32(s_tmem + 96, sb);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(sb);
        mask(sb, 96);
        fold(sb, 0);
        const float mx = fmaxf(ptx::fmax3(mx8[0], mx8[1], mx8[2]),
                               ptx::fmax3(ptx::fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        const float mnew = mx * sl;
        if (j == 0) {
          m = mnew;
        } else {
          // O is rescaled only when the running max grows by more than 2^8;
          // otherwise the old max stays the reference and P stays below 2^8.
          const bool need = mnew > m + 8.0f;
          if (__any_sync(0xffffffffu, need)) {
            const float mm = need ? mnew : m;
            const float f = ptx::ex2(m - mm);
            const uint32_t xp = x - 1;
            if (!(ok = wait_x(o_ready + (xp & 1), (xp >> 1) & 1, ctl, status, kSiteFwdSoftO, budget)))
              break;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < kD2 / 32; ++c) {
              uint32_t ov[32];
              ptx::tmem_ld32(o_tmem + 32 * c, ov);
              ptx::tmem_ld_wait();
              ptx::reg_fence32(ov);
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
              ptx::tmem_st32(o_tmem + 32 * c, ov);
            }
            ptx::tmem_st_wait();
            l *= f;
            m = mm;
          }
        }
        // a row with every key of this tile masked (possible only above the diagonal) keeps m
        const float mu = (m == -INFINITY) ? 0.f : m;
        // P = 2^(S sl - m): scale and shift on fp32 pairs, exp2 per element, sums on pairs
        const uint64_t sl2 = ptx::f2_packf(sl, sl), nmu2 = ptx::f2_packf(-mu, -mu);
        uint64_t ls2[2] = {ptx::f2_packf(0.f, 0.f), ptx::f2_packf(0.f, 0.f)};
        auto exp_store = [&](const uint32_t(&v)[32], int c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float x0, x1;
            ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(v[2 * e], v[2 * e + 1]), sl2, nmu2), x0, x1);
            const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
            ls2[e & 1] = ptx::f2_add(ls2[e & 1], ptx::f2_packf(p0, p1));
            pk[e] = ptx::pack_bf16(p0, p1);
          }
          ptx::tmem_st16(s_tmem + 16 * c, pk);
        };
        ptx::tmem_ld32(s_tmem + 64, sb);  // chunk 2 again, read while chunk 0 is exponentiated
        exp_store(sa[0], 0);
        ptx::tmem_ld32(s_tmem + 96, sa[0]);  // chunk 3 again
        exp_store(sa[1], 1);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(sb);
        ptx::reg_fence32(sa[0]);
        mask(sb, 64);
        exp_store(sb, 2);
        mask(sa[0], 96);
        exp_store(sa[0], 3);
        {
          float a0, a1, b0, b1;
          ptx::f2_unpack(ls2[0], a0, a1);
          ptx::f2_unpack(ls2[1], b0, b1);
          l += (a0 + a1) + (b0 + b1);
        }
        if (j + 1 == n) {
          // row statistics of the finished item go to the epilogue
          if (kq >= 2 &&
              !(ok = ptx::mbar_wait(ml_empty + ob, ((kq - 2) >> 1) & 1, ctl, status, kSiteFwdSoftMl, budget)))
            break;
          ml[ob * kTile + r] = make_float2(m, l);
          ptx::mbar_arrive(ml_full + ob);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        signal_p(p_full + (x & 1));
      }
      ++kq;
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 4-7, both CTAs)
    const int quarter = warp & 3;  // TMEM lanes 32 (warp % 4) .. are this warp's rows
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr float kLn2 = 0.6931471805599453f;
    auto signal_free = [&](uint64_t* bar) {
      if (lane != 0) return;
      if (!PAIR || leader)
        ptx::mbar_arrive(bar);
      else
        ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(bar), 0));
    };
    uint32_t kq = 0;
    for (int idx = cluster; idx < n_items; idx += n_clusters) {
      const FwdStreamItem I = stream_item<CAUSAL, PAIR>(p, idx, rank);
      const int qi = kTile * I.t + r;
      const bool row_ok = qi < I.Lq;
      __nv_bfloat16* orow = p.o + (I.o_row + r) * static_cast<int64_t>(p.heads) * kD2 + static_cast<int64_t>(I.h) * kD2;
      if (I.n_kv == 0) {  // no keys: O = 0, LSE = -inf
        if (row_ok) {
          for (int c = 0; c < kD2; c += 8) ptx::st_v4(orow + c, 0, 0, 0, 0);
          p.lse[I.lse0 + r] = -INFINITY;
        }
        continue;
      }
      const uint32_t ob = kq & 1;
      bool w = wait_x(o_final + ob, (kq >> 1) & 1, ctl, status, kSiteFwdEpi, budget);
      w = w && ptx::mbar_wait(ml_full + ob, (kq >> 1) & 1, ctl, status, kSiteFwdEpi, budget);
      if (!w) break;
      ptx::tc_fence_after();
      const float2 st = ml[ob * kTile + r];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ml_empty + ob);
      const float inv_l = st.y > 0.f ? 1.0f / st.y : 0.f;
      const uint32_t o_tmem = tmem + lane_base + (ob ? Lay::kColO1 : Lay::kColO0);
#pragma unroll 1
      for (int c = 0; c < kD2 / 32; ++c) {
        uint32_t ov[32];
        ptx::tmem_ld32(o_tmem + 32 * c, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(ov);
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wv[e] = ptx::pack_bf16(__uint_as_float(ov[8 * q4 + 2 * e]) * inv_l,
                                     __uint_as_float(ov[8 * q4 + 2 * e + 1]) * inv_l);
            ptx::st_v4(orow + 32 * c + 8 * q4, wv[0], wv[1], wv[2], wv[3]);
          }
        }
      }
      if (row_ok) p.lse[I.lse0 + r] = (st.x + log2f(st.y)) * kLn2;
      ptx::tc_fence_before();
      __syncwarp();
      signal_free(o_free + ob);
      ++kq;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();  // every MMA into either CTA's TMEM is done and every TMEM read finished
  if (warp == 9) {
    ptx::tc_fence_after();
    if (PAIR)
      ptx::tmem_dealloc2(tmem, Lay::kTmemCols);
    else
      ptx::tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

template <bool CAUSAL, bool PAIR>
cudaError_t launch_fwd_stream_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdStreamParams& p,
                          int grid, cudaStream_t stream) {
  using Lay = FwdStreamLayout<PAIR>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fwd_stream_kernel<CAUSAL, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kAlloc);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(320);
  cfg.dynamicSmemBytes = Lay::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = PAIR ? 2 : 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_stream_kernel<CAUSAL, PAIR>, tq, tk, tv, p);
}

}  // namespace

cudaError_t launch_fwd_stream(bool pair, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const int32_t* offsets, const int4* items, int32_t* status,
                              void* o, float* lse, int heads, int total, int bcast, int q_len, float scale,
                              uint64_t budget_ns, int grid, cudaStream_t stream) {
  FwdStreamParams p;
  p.offsets = offsets;
  p.items = items;
  p.status = status;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.heads = heads;
  p.total = total;
  p.bcast = bcast;
  p.q_len = q_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.budget_ns = budget_ns;
  if (pair)
    return causal ? launch_fwd_stream_t<true, true>(tq, tk, tv, p, grid, stream)
                  : launch_fwd_stream_t<false, true>(tq, tk, tv, p, grid, stream);
  return causal ? launch_fwd_stream_t<true, false>(tq, tk, tv, p, grid, stream)
                : launch_fwd_stream_t<false, false>(tq, tk, tv, p, grid, stream);
}

}  // namespace jfa
