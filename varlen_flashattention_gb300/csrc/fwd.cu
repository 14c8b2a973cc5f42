// Jagged FlashAttention forward on tcgen05 tensor cores (sm_103a).
//
// What it computes ("Cutting-edge isn't plug-and-play: customizing FA4 on
// B300", FlashAttention recap; "Optimizing Jagged Flash Attention with TLX",
// third paragraph): for every packed sequence and head, O = softmax(scale Q
// K^T) V and LSE = ln sum_j exp(scale q.k_j), tiled so S never reaches HBM.
//
// How (GB300 design; prior art is the TLX and FA4 kernels the pages describe):
//  * persistent grid, one CTA per SM, walking a longest-first queue of
//    (sequence, head, 128-row query tile) items built on the device;
//  * warp 4 = TMA producer: the Q tile, then K_0, K_1, V_0, K_2, V_1, ... into
//    a ring of shared-memory slots (128B-swizzled 128x64 boxes);
//  * warp 5 = MMA issuer: S_j = Q K_j^T into one of two TMEM score buffers,
//    then O += P_j V_j with P_j read from TMEM (O lives in TMEM all along);
//  * warps 0-3 = softmax: thread i owns query row i (TMEM lane i): loads its
//    score row, masks only in the peeled tail / diagonal tile, keeps a running
//    maximum that is raised (and O rescaled) only when the row maximum grows
//    by more than 2^8, writes P as bf16 over the scores in TMEM, and at the
//    end normalises O and writes O and LSE for the rows of the sequence.
//  * The score buffers double-buffer S across iterations, so S_{j+1} is on
//    the tensor core while the softmax warps work on S_j; with head_dim 192,
//    O (192 columns) plus two score buffers still fit the 512 TMEM columns.
//  * Every mbarrier wait is bounded; a wait that runs out records
//    JFA_ERR_TIMEOUT in the workspace status word and all roles leave.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "jfa_internal.h"
#include "ptx.cuh"
#include "trace.cuh"

namespace jfa {

struct FwdParams {
  const int32_t* offsets;  // self: sequence offsets; broadcast: K/V offsets
  const int4* items;
  const int4* item_seq;    // varlen: (first query row, L_q, first key row, L_k) of each item
  int32_t* status;         // status block (n_items at [2])
  __nv_bfloat16* o;
  float* lse;
  int32_t heads;
  int32_t total;           // self: rows of Q/K/V; broadcast: total_k
  int32_t bcast;
  int32_t q_len;           // broadcast only
  int32_t var, group;      // varlen: bounds from item_seq; query heads per KV head
  float scale_log2;
  uint64_t budget_ns;
  int32_t* counter;        // items handed out so far (zero at launch; causal items are claimed from it)
};

template <int D>
struct FwdLayout {
  static constexpr int kAtoms = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kSlots = (D == 64) ? 8 : (D == 128 ? 6 : 3);
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = kTileBytes;
  static constexpr int kOffBars = kTileBytes * (1 + kSlots);
  static constexpr int kRing = 8;  // claimed items in flight (causal)
  // q_full, q_empty, slot_full[S], slot_empty[S], s_full[2], p_full[2], o_ready[2], o_free, drain,
  // ring_full[R], ring_empty[R]
  static constexpr int kNumBars = 2 + 2 * kSlots + 2 + 2 + 2 + 1 + 1 + 2 * kRing;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kOffRing = kOffMisc + 64;  // item index of each ring entry
  static constexpr int kBytes = kOffRing + kRing * 4;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColO + D <= kTmemCols, "TMEM budget");
};

struct FwdItem {
  int b, h, t;
  int hk;         // KV head read by query head h
  int delta;      // L_k - L_q: key j is visible to query i iff j <= i + delta (causal)
  int q_tma_row;  // row of the Q tile in the Q tensor map
  int kv_row0;    // first K/V row of the sequence
  int Lq, Lk;
  int n_kv;       // K/V tiles to visit
  int64_t o_row;  // first output row of the tile ([rows, H, D] view of O)
  int64_t lse0;   // index of the tile's first LSE entry
};

template <bool CAUSAL>
__device__ __forceinline__ FwdItem fwd_item(const FwdParams& p, int idx) {
  const int4 it = p.items[idx];
  FwdItem I;
  I.b = it.x;
  I.h = it.y;
  I.t = it.z;
  if (p.var) {
    const int4 sq = p.item_seq[idx];
    I.Lq = sq.y;
    I.Lk = sq.w;
    I.kv_row0 = sq.z;
    I.hk = I.h / p.group;
    I.delta = I.Lk - I.Lq;
    I.q_tma_row = sq.x + kTile * I.t;
    I.o_row = I.q_tma_row;
    I.lse0 = static_cast<int64_t>(I.h) * p.total + I.q_tma_row;
    I.n_kv = it.w;  // the queue's cost: key tiles visited
    return I;
  }
  I.hk = I.h;
  I.delta = 0;
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
  I.n_kv = CAUSAL ? min(I.t + 1, nk) : nk;
  return I;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(192, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using Lay = FwdLayout<D>;
  constexpr int kSlots = Lay::kSlots;
  constexpr uint32_t kIdescQK = ptx::idesc_bf16(128, 128, false, false);
  constexpr uint32_t kIdescPV = ptx::idesc_bf16(128, D, false, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBars);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* slot_full = bars + 2;
  uint64_t* slot_empty = bars + 2 + kSlots;
  uint64_t* s_full = bars + 2 + 2 * kSlots;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_ready = p_full + 2;
  uint64_t* o_free = o_ready + 2;
  uint64_t* drain = o_free + 1;
  // Causal items cost 1 .. n key tiles, very unequal even in longest-first
  // order: the producer claims them on demand from an atomic counter and
  // passes each index to the MMA thread and the softmax warps through a ring
  // (an index of -1 ends the stream). Other items are dealt round-robin.
  uint64_t* ring_full = drain + 1;
  uint64_t* ring_empty = ring_full + Lay::kRing;
  int32_t* ring_idx = reinterpret_cast<int32_t*>(smem + Lay::kOffRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  ptx::CtaCtl* ctl = reinterpret_cast<ptx::CtaCtl*>(smem + Lay::kOffMisc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    for (int i = 0; i < kSlots; ++i) {
      ptx::mbar_init(slot_full + i, 1);
      ptx::mbar_init(slot_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(s_full + i, 1);
      ptx::mbar_init(p_full + i, 4);
      ptx::mbar_init(o_ready + i, 1);
    }
    ptx::mbar_init(o_free, 4);
    ptx::mbar_init(drain, 1);
    for (int i = 0; i < Lay::kRing; ++i) {
      ptx::mbar_init(ring_full + i, 1);
      ptx::mbar_init(ring_empty + i, 5);  // the MMA thread and the four softmax warps
    }
    ctl->abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
  }
  if (warp == 5) {
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
  // The next item index of a consumer (the MMA thread, or a whole softmax
  // warp whose lane 0 gives the entry back): from the ring when causal,
  // else the round-robin share st. -1 at the end of the stream, -2 when the
  // wait gave up.
  auto take_idx = [&](uint32_t k, int& st, bool warp_wide) -> int {
    if constexpr (!CAUSAL) {
      const int v = st;
      st += gridDim.x;
      return v < n_items ? v : -1;
    }
    const uint32_t e = k % Lay::kRing;
    bool w = ptx::mbar_wait(ring_full + e, (k / Lay::kRing) & 1, ctl, status, kSiteFwdMmaQ, budget);
    if (warp_wide) w = ptx::warp_all(w);
    if (!w) return -2;
    const int v = ring_idx[e];
    if (warp_wide) {
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ring_empty + e);
    } else {
      ptx::mbar_arrive(ring_empty + e);
    }
    return v;
  };

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t pos = 0, kq = 0;
      bool ok = true;
      auto load_tile = [&](const CUtensorMap* map, int h, int row) -> bool {
        const uint32_t slot = pos % kSlots, round = pos / kSlots;
        if (!ptx::mbar_wait(slot_empty + slot, (round & 1) ^ 1, ctl, status, kSiteFwdProdSlot, budget)) return false;
        uint8_t* dst = smem + Lay::kOffSlots + slot * Lay::kTileBytes;
        ptx::mbar_arrive_expect_tx(slot_full + slot, Lay::kTileBytes);
#pragma unroll
        for (int a = 0; a < Lay::kAtoms; ++a) ptx::tma_load_2d(dst + a * 16384, map, slot_full + slot, h * D + 64 * a, row);
        ++pos;
        return true;
      };
      uint32_t kc = 0;  // items claimed
      auto claim = [&]() -> int {  // next item index, -1 at the end, -2 when a wait gave up
        if constexpr (!CAUSAL) {
          const int v = static_cast<int>(blockIdx.x + kc++ * gridDim.x);
          return v < n_items ? v : -1;
        }
        const uint32_t e = kc % Lay::kRing;
        if (!ptx::mbar_wait(ring_empty + e, ((kc / Lay::kRing) & 1) ^ 1, ctl, status, kSiteFwdProdQ, budget))
          return -2;
        int v = atomicAdd(p.counter, 1);
        if (v >= n_items) v = -1;
        ring_idx[e] = v;
        ptx::mbar_arrive(ring_full + e);  // release: the index is visible to the entry's waiters
        ++kc;
        return v;
      };
      for (int idx = claim(); ok && idx >= 0; idx = claim()) {
        const FwdItem I = fwd_item<CAUSAL>(p, idx);
        if (I.n_kv == 0) continue;
        // debug builds: the Q tile and every K/V tile start inside their sequences and heads
        if (!JFA_TILE_OK(I.t >= 0 && kTile * I.t < I.Lq && I.h >= 0 && I.h < p.heads, ctl, status, kSiteCheckFwdQ))
          break;
        if (!JFA_TILE_OK(I.n_kv > 0 && kTile * (I.n_kv - 1) < I.Lk && I.hk >= 0, ctl, status, kSiteCheckFwdKV)) break;
        if (!ptx::mbar_wait(q_empty, (kq & 1) ^ 1, ctl, status, kSiteFwdProdQ, budget)) break;
        ptx::mbar_arrive_expect_tx(q_full, Lay::kTileBytes);
#pragma unroll
        for (int a = 0; a < Lay::kAtoms; ++a)
          ptx::tma_load_2d(smem + Lay::kOffQ + a * 16384, &tm_q, q_full, I.h * D + 64 * a, I.q_tma_row);
        ok = load_tile(&tm_k, I.hk, I.kv_row0);
        for (int j = 0; ok && j < I.n_kv; ++j) {
          if (j + 1 < I.n_kv) ok = load_tile(&tm_k, I.hk, I.kv_row0 + kTile * (j + 1));
          if (ok) ok = load_tile(&tm_v, I.hk, I.kv_row0 + kTile * j);
        }
        ++kq;
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t pos = 0, kq = 0, it = 0;  // ring position, items done, KV iterations done
      const uint32_t q_addr = ptx::smem_u32(smem + Lay::kOffQ);
      bool ok = true;
      auto slot_wait = [&](uint32_t& slot) -> bool {
        slot = pos % kSlots;
        const uint32_t round = pos / kSlots;
        if (!ptx::mbar_wait(slot_full + slot, round & 1, ctl, status, kSiteFwdMmaSlot, budget)) return false;
        ptx::tc_fence_after();
        return true;
      };
      auto issue_qk = [&](uint32_t slot, uint32_t x) {
        const uint32_t k_addr = ptx::smem_u32(smem + Lay::kOffSlots + slot * Lay::kTileBytes);
        const uint32_t d_tmem = tmem + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          ptx::mma_ss(d_tmem, ptx::sdesc_sw128(q_addr + off, 16, 1024), ptx::sdesc_sw128(k_addr + off, 16, 1024),
                      kIdescQK, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(s_full + (x & 1));
        ptx::mma_commit(slot_empty + slot);
        ++pos;
      };
      uint32_t kr = 0;
      int st = blockIdx.x;
      for (int idx = take_idx(kr++, st, false); ok && idx >= 0; idx = take_idx(kr++, st, false)) {
        const FwdItem I = fwd_item<CAUSAL>(p, idx);
        const int n = I.n_kv;
        if (n == 0) continue;
        if (!ptx::mbar_wait(q_full, kq & 1, ctl, status, kSiteFwdMmaQ, budget)) break;
        ptx::tc_fence_after();
        uint32_t slot;
        if (!(ok = slot_wait(slot))) break;
        issue_qk(slot, it);
        if (n == 1) ptx::mma_commit(q_empty);
        for (int j = 0; ok && j < n; ++j) {
          const uint32_t x = it + j;
          if (j + 1 < n) {
            if (!(ok = slot_wait(slot))) break;
            issue_qk(slot, x + 1);
            if (j + 2 == n) ptx::mma_commit(q_empty);
          }
          if (!(ok = ptx::mbar_wait(p_full + (x & 1), (x >> 1) & 1, ctl, status, kSiteFwdMmaP, budget))) break;
          if (j == 0 && kq > 0) {
            if (!(ok = ptx::mbar_wait(o_free, (kq - 1) & 1, ctl, status, kSiteFwdMmaOFree, budget))) break;
          }
          if (!(ok = slot_wait(slot))) break;
          ptx::tc_fence_after();
          const uint32_t v_addr = ptx::smem_u32(smem + Lay::kOffSlots + slot * Lay::kTileBytes);
          const uint32_t p_tmem = tmem + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            ptx::mma_ts(tmem + Lay::kColO, p_tmem + kk * 8, ptx::sdesc_sw128(v_addr + kk * 2048, 16384, 1024),
                        kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(o_ready + (x & 1));
          ptx::mma_commit(slot_empty + slot);
          ++pos;
        }
        it += n;
        ++kq;
      }
      // make sure nothing issued is still running when TMEM is released
      ptx::mma_commit(drain);
      ptx::CtaCtl no_abort{0, 0};
      ptx::mbar_wait(drain, 0, &no_abort, nullptr, kSiteFwdDrain, budget);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue (warps 0-3)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row of the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl = p.scale_log2;
    constexpr float kLn2 = 0.6931471805599453f;
    uint32_t it = 0, kq = 0, kr = 0;
    int st = blockIdx.x;
    for (int idx = take_idx(kr++, st, true); idx >= 0; idx = take_idx(kr++, st, true)) {
      const FwdItem I = fwd_item<CAUSAL>(p, idx);
      const int n = I.n_kv;
      const bool row_ok = kTile * I.t + r < I.Lq;
      __nv_bfloat16* orow = p.o + (I.o_row + r) * static_cast<int64_t>(p.heads) * D + static_cast<int64_t>(I.h) * D;
      if (n == 0) {  // no visible key: O = 0, LSE = -inf
        if (row_ok) {
          for (int c = 0; c < D; c += 8) ptx::st_v4(orow + c, 0, 0, 0, 0);
          p.lse[I.lse0 + r] = -INFINITY;
        }
        continue;
      }
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const uint32_t x = it + j;
        const uint32_t s_tmem = tmem + lane_base + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
        if (!(ok = ptx::mbar_wait(s_full + (x & 1), (x >> 1) & 1, ctl, status, kSiteFwdSoftS, budget))) break;
        ptx::tc_fence_after();
        uint32_t sv[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32(s_tmem + 32 * c, sv[c]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::reg_fence32(sv[c]);
        // peeled tail: only tiles that cross the (bottom-right aligned) diagonal
        // or the end of the keys are masked
        const bool tail = (CAUSAL && kTile * j + kTile - 1 > kTile * I.t + I.delta) || kTile * (j + 1) > I.Lk;
        if (tail) {
          const int lim = CAUSAL ? min(r + 1 + kTile * (I.t - j) + I.delta, I.Lk - kTile * j) : I.Lk - kTile * j;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e >= lim) sv[c][e] = __float_as_uint(-INFINITY);
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(sv[c][e]));
        const float mnew = mx * sl;
        if (j == 0) {
          m = mnew;
        } else {
          const bool need = mnew > m + 8.0f;
          if (__any_sync(0xffffffffu, need)) {
            const float mm = need ? mnew : m;
            const float f = ptx::ex2(m - mm);
            const uint32_t xp = x - 1;
            if (!(ok = ptx::mbar_wait(o_ready + (xp & 1), (xp >> 1) & 1, ctl, status, kSiteFwdSoftO, budget))) break;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t ov[32];
              ptx::tmem_ld32(tmem + lane_base + Lay::kColO + 32 * c, ov);
              ptx::tmem_ld_wait();
              ptx::reg_fence32(ov);
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
              ptx::tmem_st32(tmem + lane_base + Lay::kColO + 32 * c, ov);
            }
            ptx::tmem_st_wait();
            l *= f;
            m = mm;
          }
        }
        // P = 2^(s*scale*log2e - m), written as bf16 pairs over the scores; a
        // row that sees no key so far (m = -inf) shifts by 0 and gets P = 0
        const float mu = (m == -INFINITY) ? 0.f : m;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ptx::ex2(fmaf(__uint_as_float(sv[c][2 * e]), sl, -mu));
            const float p1 = ptx::ex2(fmaf(__uint_as_float(sv[c][2 * e + 1]), sl, -mu));
            l += p0 + p1;
            pk[e] = ptx::pack_bf16(p0, p1);
          }
          ptx::tmem_st16(s_tmem + 16 * c, pk);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full + (x & 1));
      }
      if (!ok) break;
      // epilogue: O / l and LSE for the rows that belong to the sequence
      const uint32_t xl = it + n - 1;
      if (!ptx::mbar_wait(o_ready + (xl & 1), (xl >> 1) & 1, ctl, status, kSiteFwdSoftO, budget)) break;
      ptx::tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;  // a row that sees no key: O = 0
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        ptx::tmem_ld32(tmem + lane_base + Lay::kColO + 32 * c, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(ov);
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = ptx::pack_bf16(__uint_as_float(ov[8 * q4 + 2 * e]) * inv_l,
                                    __uint_as_float(ov[8 * q4 + 2 * e + 1]) * inv_l);
            ptx::st_v4(orow + 32 * c + 8 * q4, w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (row_ok) p.lse[I.lse0 + r] = (m + log2f(l)) * kLn2;
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(o_free);
      it += n;
      ++kq;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

// ------------------------------------------------------------------ launcher

template <int D, bool CAUSAL>
static cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdParams& p, int grid, cudaStream_t stream) {
  using Lay = FwdLayout<D>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(fwd_kernel<D, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kAlloc);
  });
  if (e != cudaSuccess) return e;
  return launch_after(fwd_kernel<D, CAUSAL>, dim3(grid), dim3(192), Lay::kAlloc, stream, tq, tk, tv, p);
}

cudaError_t launch_fwd(int head_dim, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const int32_t* offsets, const int4* items, const int4* item_seq, const VarInfo& var,
                       int32_t* status, void* o, float* lse, int heads,
                       int total, int bcast, int q_len, float scale, uint64_t budget_ns, int grid,
                       cudaStream_t stream) {
  FwdParams p;
  p.offsets = offsets;
  p.items = items;
  p.status = status;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.heads = heads;
  p.total = total;
  p.bcast = bcast;
  p.q_len = q_len;
  p.item_seq = item_seq;
  p.var = var.var;
  p.group = var.group;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.budget_ns = budget_ns;
  p.counter = status + kStatusItemCounter;
  if (head_dim == 64) return causal ? launch_fwd_t<64, true>(tq, tk, tv, p, grid, stream)
                                    : launch_fwd_t<64, false>(tq, tk, tv, p, grid, stream);
  if (head_dim == 128) return causal ? launch_fwd_t<128, true>(tq, tk, tv, p, grid, stream)
                                     : launch_fwd_t<128, false>(tq, tk, tv, p, grid, stream);
  if (head_dim == 192) return causal ? launch_fwd_t<192, true>(tq, tk, tv, p, grid, stream)
                                     : launch_fwd_t<192, false>(tq, tk, tv, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace jfa
