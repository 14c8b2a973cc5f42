// Jagged FlashAttention backward on tcgen05 tensor cores (sm_103a).
//
// What it computes ("Cutting-edge isn't plug-and-play: customizing FA4 on
// B300", Phase 2 and its pseudocode): for each tile pair, S and dP are rebuilt
// from Q, K, V, dO; P comes from S and the LSE saved by the forward; then
//   D = rowsum(dO * O) ("delta"), dS = P * (dP - D),
//   dV += P^T dO, dK += scale dS^T Q, dQ += scale dS K.
// Broadcast-Q ("Optimizing Jagged Flash Attention with TLX", third
// paragraph): every sequence reads the same Q, so dQ sums over the batch.
// Head-axis chunking (TwelveLabs Phase 2): with head_dim 192 one pass owns a
// 64-wide slice c of dQ/dK/dV, while S and dP are still accumulated over all
// of the head dimension (three passes rebuild S and dP).
//
// Kernel organisation (GB300 design):
//  * persistent grid; items are (sequence, head, 128-row K/V tile[, slice])
//    from the longest-first queue; K and V stay in shared memory for the item
//    while the producer streams the Q, dO tiles (and their LSE/delta rows)
//    of every query tile that sees this K/V tile;
//  * scores are computed transposed, S^T = K Q^T, so TMEM lane = key row and
//    P^T can feed dV += P^T dO straight from TMEM;
//  * warps 0-7 (one thread per key row; warps w and w + 4 share the TMEM lanes
//    of their rows, warps 0-3 take query columns 0-63 and warps 4-7 columns
//    64-127: the exp loops are latency-bound, and two warps per SM
//    sub-partition run them almost twice as fast while the tensor core is
//    busy) turn S^T into P^T (bf16, packed over the S^T columns each group has
//    read) and dP^T into dS^T (bf16, written to shared memory in the
//    128B-swizzled layout the tensor core reads as dS for dQ and as dS^T for
//    dK; with a single stage also packed into TMEM over the dP^T columns each
//    group has read, as dS^T for dK);
//  * warps 10-13 drain dQ from TMEM into an fp32 accumulator (the cross-CTA
//    reduction; contended in broadcast-Q) and write dK and dV at the end of
//    each item. dQ is staged, in 128B-swizzled fp32 boxes, in the dO stage
//    buffer of its own query tile (free once the dQ MMA has completed: dV was
//    its last reader), a stage-sized part at a time (with a single stage,
//    head_dim 192, in the dS buffer instead) and added by TMA reduce-add
//    ("Optimizing Jagged Flash Attention with TLX", fifth paragraph: staging
//    of the dQ reduce-add); the drain warps release the stage to the producer
//    after TMA has read it; the Q half of the stage is released by the MMA
//    warp right after dK, so the next query tile's Q never waits for dQ. Per-thread vector atomics measured slower: their
//    strided requests held the SM's load/store path that the softmax warps
//    use for TMEM and shared memory;
//  * warp 8 = TMA producer, warp 9 = MMA issuer; 448 threads, so a thread has
//    at most 128 registers.
//  * Order inside one query tile: dP^T, dV, dQ, [S^T of the next tile], dK:
//    dQ goes first so that its drain runs under the S^T and dK MMAs, and the
//    softmax of the next tile overlaps dK. With a single Q/dO stage (head_dim
//    192) S^T is issued at the start of its own tile (TwelveLabs, bug hunting:
//    the single-stage deadlock) and dK (from TMEM) precedes dQ. That stage is
//    tracked per 64-column atom: a pass over slice c needs atom c of Q and dO
//    again (dK, dV) but the other atoms only for S^T and dP^T, so those are
//    released when S^T / dP^T complete and the next tile's copies of them load
//    while dV, dK and dQ run; S^T and dP^T consume atom c last.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "jfa_internal.h"
#include "ptx.cuh"
#include "trace.cuh"

namespace jfa {

struct BwdParams {
  const int32_t* offsets;     // self: sequence offsets; broadcast: K/V offsets
  const int32_t* tile_base;   // self: padded q-tile index of each sequence
  const int4* items;
  const int4* item_seq;       // (first row, length, tile_base) of each item's sequence
  int32_t* status;
  const float* lse2p;         // -LSE log2(e), tile-padded (stored negated)
  const float* deltap;        // -delta, tile-padded (stored negated)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int32_t heads, total, bcast, q_len, causal, n_chunks;
  int32_t col0;               // first head-dim column of this launch's slices (slice c: col0 + c DC ..)
  int32_t chunk;              // DC, the slice width
  int32_t pad_tiles;          // self, varlen: query tiles per head in the padded arrays
  int32_t var, group;         // varlen: items carry query and key bounds; query heads per KV head
  int32_t kv_heads;           // heads of K, V, dK, dV
  float scale, scale_log2;
  uint64_t budget_ns;
};

template <int D, int DC>
struct BwdLayout {
  static constexpr int kAtoms = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = (D == 192) ? 1 : 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;                       // kStages x Q
  static constexpr int kOffDO = kOffQ + kStages * kTileBytes;         // kStages x dO
  static constexpr int kOffDS = kOffDO + kStages * kTileBytes;        // 128 x 128 bf16
  static constexpr int kOffRow = kOffDS + kTile * kTile * 2;          // kStages x (lse2[128], delta[128])
  static constexpr int kOffBars = kOffRow + kStages * 1024;
  // With one stage, Q and dO are tracked per 64-column atom (barrier i = atom i), so the atoms
  // outside the pass's slice can be refilled as soon as S^T / dP^T have read them.
  static constexpr int kQBars = (kStages == 1) ? kAtoms : kStages;
  // k_full, k_empty, v_full, v_empty, q_full[B], q_empty[B], do_full[B], do_empty[B], s_full, p_full,
  // dp_full, ds_full, ds_free, dq_full, dq_free, acc_full, acc_free, drain, staged, stage_read, stage_free
  static constexpr int kNumBars = 4 + 4 * kQBars + 13;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64;
  static constexpr int kAlloc = kBytes + 256;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + DC;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColDK + DC <= kTmemCols, "TMEM budget");
  static_assert(kAlloc <= 232448, "shared memory budget");
};

struct BwdItem {
  int b, h, t, c;  // sequence, (KV) head, K/V tile, head-dim slice
  int hq0;         // first query head that reads KV head h (varlen: h * group; else h)
  int nqt;         // query tiles per query head; the item's steps are nq = group * nqt
  int delta;       // L_k - L_q: key j is visible to query i iff j <= i + delta (causal)
  int kv_row0;     // first K/V row of the tile
  int Lk, Lq;
  int i0, nq;      // query tiles i0 .. i0+nq-1
  int q_row0;      // Q row of query tile 0 (TMA)
  int do_row0;     // dO row of query tile 0 (TMA)
  int64_t row_base;  // padded LSE/delta index of query tile 0 (times 128)
};

// An item's record: two independent loads (the queue stores each item's
// sequence start, length and tile base beside it), no dependent lookup.
__device__ __forceinline__ BwdItem bwd_item(const BwdParams& p, int v) {
  const int idx = v / p.n_chunks;
  BwdItem I;
  I.c = v - idx * p.n_chunks;
  const int4 it = p.items[idx];
  const int4 sq = p.item_seq[idx];
  I.b = it.x;
  I.h = it.y;
  I.t = it.z;
  const int s0 = sq.x;
  I.Lk = sq.y;
  I.kv_row0 = s0 + kTile * I.t;
  I.hq0 = I.h;
  I.delta = 0;
  if (p.var) {  // item_seq: (first query row, L_q, first key row, L_k); items.w: query tile base
    I.Lq = sq.y;
    I.Lk = sq.w;
    I.kv_row0 = sq.z + kTile * I.t;
    I.q_row0 = s0;
    I.do_row0 = s0;
    I.hq0 = I.h * p.group;
    I.delta = I.Lk - I.Lq;
    I.row_base = (static_cast<int64_t>(I.hq0) * p.pad_tiles + it.w) * kTile;
    const int nq = (I.Lq + kTile - 1) / kTile;
    const int i_min = p.causal ? max(0, kTile * I.t - I.delta) : 0;  // first query that sees the tile
    I.i0 = i_min / kTile;
    I.nqt = i_min < I.Lq ? nq - I.i0 : 0;
    I.nq = p.group * I.nqt;
    return I;
  }
  if (!p.bcast) {
    I.Lq = I.Lk;
    I.q_row0 = s0;
    I.do_row0 = s0;
    I.row_base = (static_cast<int64_t>(I.h) * p.pad_tiles + sq.z) * kTile;
  } else {
    I.Lq = p.q_len;
    I.q_row0 = 0;
    I.do_row0 = I.b * p.q_len;
    const int nqt = (p.q_len + kTile - 1) / kTile;
    I.row_base = ((static_cast<int64_t>(I.b) * p.heads + I.h) * nqt) * kTile;
  }
  const int nq = (I.Lq + kTile - 1) / kTile;
  I.i0 = p.causal ? I.t : 0;
  I.nq = nq - I.i0;
  I.nqt = I.nq;
  return I;
}

// Step ii of an item: query head hq0 + g, query tile i. The steps run over the
// query tiles of each query head of the group in turn.
__device__ __forceinline__ void bwd_step(const BwdItem& I, int ii, int& g, int& i) {
  g = (I.nqt == I.nq) ? 0 : ii / I.nqt;
  i = I.i0 + ii - g * I.nqt;
}

// First head-dim column of an item's slice (0 when one slice covers the head).
template <int D, int DC>
__device__ __forceinline__ int slice_col(const BwdParams& p, const BwdItem& I) {
  if constexpr (DC == D) return 0;
  else return p.col0 + I.c * DC;
}

// One-stage pipeline: the n-th 64-column atom of Q (or dO) in load and MMA
// order for a pass over the slice of `sa` atoms starting at atom ca: the atoms
// outside the slice in ascending order, then the slice's. S^T (dP^T) reads
// every atom but only dK (dV) reads the slice again, so the others are refilled
// for the next query tile while this one finishes.
__device__ __forceinline__ int atom_at(int n, int ca, int sa, int atoms) {
  return n < atoms - sa ? (n < ca ? n : n + sa) : ca + (n - (atoms - sa));
}

template <int D, int DC>
__global__ void __launch_bounds__(448, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
               const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using Lay = BwdLayout<D, DC>;
  constexpr int kSt = Lay::kStages;
  constexpr int kSliceAtoms = DC / 64;  // 64-column atoms of one head-dim slice
  constexpr uint32_t kIdS = ptx::idesc_bf16(128, 128, false, false);   // S^T, dP^T
  constexpr uint32_t kIdAcc = ptx::idesc_bf16(128, DC, false, true);   // dV, dK
  constexpr uint32_t kIdDQ = ptx::idesc_bf16(128, DC, true, true);     // dQ (A = dS, M-major)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the layout needs a 1024-byte aligned base; the launch reserves 256 bytes of slack
  if (smem + Lay::kBytes > smem_raw + Lay::kAlloc) {
    wait_prior_grid();  // the status block was cleared before this kernel
    if (threadIdx.x == 0) atomicCAS(p.status, JFA_OK, JFA_ERR_UNSUPPORTED);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBars);
  // K and V of an item are released separately: V after the item's last dP^T,
  // K after its last dQ, so the next item's V (and most of its K) load while
  // the last tile of this one is still computing
  uint64_t* k_full = bars + 0;
  uint64_t* k_empty = bars + 1;
  uint64_t* v_full = bars + 2;
  uint64_t* v_empty = bars + 3;
  // per stage (two stages) or per 64-column atom (one stage)
  constexpr int kQB = Lay::kQBars;
  uint64_t* q_full = bars + 4;            // Q and the LSE / delta rows of a query tile
  uint64_t* q_empty = bars + 4 + kQB;
  uint64_t* do_full = bars + 4 + 2 * kQB;  // dO of a query tile
  uint64_t* do_empty = bars + 4 + 3 * kQB;
  uint64_t* s_full = bars + 4 + 4 * kQB;
  uint64_t* p_full = s_full + 1;
  uint64_t* dp_full = s_full + 2;
  uint64_t* ds_full = s_full + 3;
  uint64_t* ds_free = s_full + 4;
  uint64_t* dq_full = s_full + 5;
  uint64_t* dq_free = s_full + 6;
  uint64_t* acc_full = s_full + 7;
  uint64_t* acc_free = s_full + 8;
  uint64_t* drain = s_full + 9;
  uint64_t* staged = s_full + 10;      // the drain threads have written (part of) the dQ staging
  uint64_t* stage_read = s_full + 11;  // TMA has read a staging round (before the next round is written)
  uint64_t* stage_free = s_full + 12;  // dS-buffer staging (one stage): TMA has read the whole tile
  // where dQ is staged: the tile's own dO stage buffer (two stages) or the dS buffer (one)
  constexpr bool kStageInDO = kSt > 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
  ptx::CtaCtl* ctl = reinterpret_cast<ptx::CtaCtl*>(smem + Lay::kOffMisc + 8);

  if (threadIdx.x == 0) {
    ptx::mbar_init(k_full, 1);
    ptx::mbar_init(k_empty, 1);
    ptx::mbar_init(v_full, 1);
    ptx::mbar_init(v_empty, 1);
    for (int i = 0; i < kQB; ++i) {
      ptx::mbar_init(q_full + i, 1);
      ptx::mbar_init(q_empty + i, 1);
      ptx::mbar_init(do_full + i, 1);
      ptx::mbar_init(do_empty + i, 1);
    }
    ptx::mbar_init(s_full, 1);
    ptx::mbar_init(p_full, 8);
    ptx::mbar_init(dp_full, 1);
    ptx::mbar_init(ds_full, 8);
    ptx::mbar_init(ds_free, 1);
    ptx::mbar_init(dq_full, 1);
    ptx::mbar_init(dq_free, 4);
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(acc_free, 4);
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(staged, 128);
    ptx::mbar_init(stage_read, 1);
    ptx::mbar_init(stage_free, 1);
    ctl->abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_do);
    ptx::prefetch_tmap(&tm_dq);
    ptx::prefetch_tmap(&tm_dk);
    ptx::prefetch_tmap(&tm_dv);
  }
  if (warp == 9) {
    ptx::tmem_alloc(tmem_slot, Lay::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // everything above is local set-up; the queue and the pre-pass are read below.
  // The post-pass is not let in early: its blocks would wait on these SMs
  // through the whole kernel.
  wait_prior_grid();
  const uint32_t tmem = *tmem_slot;
  const int n_work = p.status[2] * p.n_chunks;
  int32_t* status = p.status;
  const uint64_t budget = p.budget_ns;
  trace::Writer tw;  // records only in a JFA_TRACE build
  tw.open(status, warp);

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // Order: the first query tile of the next item (its stage frees two tiles
    // before the end of the current item) before that item's K and V (which
    // wait for the last MMA of the current item), then its later query tiles.
    if (lane == 0) {
      uint32_t pos = 0, kitem = 0;
      uint32_t nq_loads[Lay::kAtoms] = {}, ndo_loads[Lay::kAtoms] = {};  // one stage: fills of each atom
      bool ok = true;
      auto next_item = [&](int v, BwdItem& I) -> int {  // next item with query tiles, from index v
        for (; v < n_work; v += gridDim.x) {
          I = bwd_item(p, v);
          if (I.nq > 0) break;
        }
        return v;
      };
      auto load_qdo = [&](const BwdItem& I, int ii) -> bool {
        int g, i;
        bwd_step(I, ii, g, i);
        if (!JFA_TILE_OK(i >= I.i0 && kTile * i < I.Lq && g >= 0 && I.hq0 + g < p.heads, ctl, status,
                         kSiteCheckBwdQ))
          return false;
        tw.rec(trace::kBwd, trace::kBwdQLoad, pos);
        const int qcol = (I.hq0 + g) * D;
        const int ca = slice_col<D, DC>(p, I) >> 6;  // first atom of the item's slice
        const int64_t rbase = I.row_base + static_cast<int64_t>(g) * p.pad_tiles * kTile;
        if constexpr (kSt == 1) {
          // per atom, in the order the MMAs release them: Q and dO atoms outside
          // slice c, dO atom c (read last by dV), Q atom c with the LSE / delta
          // rows (read last by dK; the softmax is done with the rows by then)
          const uint32_t par = (pos & 1) ^ 1;
          const int qrow = I.q_row0 + kTile * i, drow = I.do_row0 + kTile * i;
          auto load_atom = [&](uint64_t* full, uint64_t* empty, uint32_t* count, const CUtensorMap* map,
                               int off, int a, int row, uint32_t extra) -> bool {
            if (!ptx::mbar_wait(empty + a, par, ctl, status, kSiteBwdProdQ, budget)) return false;
            ptx::mbar_arrive_expect_tx(full + a, 16384 + extra);
            ptx::tma_load_2d(smem + off + a * 16384, map, full + a, qcol + 64 * a, row);
            ++count[a];
            return true;
          };
          constexpr int kOut = Lay::kAtoms - kSliceAtoms;  // atoms outside the slice
#pragma unroll 1
          for (int n = 0; n < kOut; ++n)
            if (!load_atom(q_full, q_empty, nq_loads, &tm_q, Lay::kOffQ, atom_at(n, ca, kSliceAtoms, Lay::kAtoms),
                           qrow, 0))
              return false;
#pragma unroll 1
          for (int n = 0; n < kOut; ++n)
            if (!load_atom(do_full, do_empty, ndo_loads, &tm_do, Lay::kOffDO,
                           atom_at(n, ca, kSliceAtoms, Lay::kAtoms), drow, 0))
              return false;
#pragma unroll 1
          for (int k = 0; k < kSliceAtoms; ++k)
            if (!load_atom(do_full, do_empty, ndo_loads, &tm_do, Lay::kOffDO, ca + k, drow, 0)) return false;
          const int last = ca + kSliceAtoms - 1;  // the last Q atom carries the LSE / delta rows
#pragma unroll 1
          for (int k = 0; k < kSliceAtoms; ++k)
            if (!load_atom(q_full, q_empty, nq_loads, &tm_q, Lay::kOffQ, ca + k, qrow, ca + k == last ? 1024 : 0))
              return false;
          uint8_t* rows = smem + Lay::kOffRow;
          ptx::bulk_load(rows, p.lse2p + rbase + static_cast<int64_t>(kTile) * i, 512, q_full + last);
          ptx::bulk_load(rows + 512, p.deltap + rbase + static_cast<int64_t>(kTile) * i, 512, q_full + last);
          ++pos;
          return true;
        }
        const uint32_t st = pos % kSt, round = pos / kSt;
        if (!ptx::mbar_wait(q_empty + st, (round & 1) ^ 1, ctl, status, kSiteBwdProdQ, budget)) return false;
        ptx::mbar_arrive_expect_tx(q_full + st, Lay::kTileBytes + 1024);
        uint8_t* qd = smem + Lay::kOffQ + st * Lay::kTileBytes;
#pragma unroll
        for (int a = 0; a < Lay::kAtoms; ++a)
          ptx::tma_load_2d(qd + a * 16384, &tm_q, q_full + st, qcol + 64 * a, I.q_row0 + kTile * i);
        uint8_t* rows = smem + Lay::kOffRow + st * 1024;
        ptx::bulk_load(rows, p.lse2p + rbase + static_cast<int64_t>(kTile) * i, 512, q_full + st);
        ptx::bulk_load(rows + 512, p.deltap + rbase + static_cast<int64_t>(kTile) * i, 512, q_full + st);
        if (!ptx::mbar_wait(do_empty + st, (round & 1) ^ 1, ctl, status, kSiteBwdProdQ, budget)) return false;
        ptx::mbar_arrive_expect_tx(do_full + st, Lay::kTileBytes);
        uint8_t* dd = smem + Lay::kOffDO + st * Lay::kTileBytes;
#pragma unroll
        for (int a = 0; a < Lay::kAtoms; ++a)
          ptx::tma_load_2d(dd + a * 16384, &tm_do, do_full + st, qcol + 64 * a, I.do_row0 + kTile * i);
        ++pos;
        return true;
      };
      BwdItem I;
      int v = next_item(blockIdx.x, I);
      if (v < n_work) ok = load_qdo(I, 0);
      while (ok && v < n_work) {
        ok = JFA_TILE_OK(I.t >= 0 && kTile * I.t < I.Lk && I.h >= 0 && I.h < p.kv_heads, ctl, status, kSiteCheckBwdKV);
        if (!ok) break;
        // V first: the previous item's last dP^T released it before its last dQ released K
        if (!(ok = ptx::mbar_wait(v_empty, (kitem & 1) ^ 1, ctl, status, kSiteBwdProdKV, budget))) break;
        ptx::mbar_arrive_expect_tx(v_full, Lay::kTileBytes);
#pragma unroll
        for (int a = 0; a < Lay::kAtoms; ++a)
          ptx::tma_load_2d(smem + Lay::kOffV + a * 16384, &tm_v, v_full, I.h * D + 64 * a, I.kv_row0);
        if (!(ok = ptx::mbar_wait(k_empty, (kitem & 1) ^ 1, ctl, status, kSiteBwdProdKV, budget))) break;
        ptx::mbar_arrive_expect_tx(k_full, Lay::kTileBytes);
#pragma unroll
        for (int a = 0; a < Lay::kAtoms; ++a)
          ptx::tma_load_2d(smem + Lay::kOffK + a * 16384, &tm_k, k_full, I.h * D + 64 * a, I.kv_row0);
        tw.rec(trace::kBwd, trace::kBwdKVLoad, kitem);
        for (int ii = 1; ok && ii < I.nq; ++ii) ok = load_qdo(I, ii);
        if (!ok) break;
        BwdItem N;
        v = next_item(v + gridDim.x, N);
        if (v < n_work) ok = load_qdo(N, 0);
        I = N;
        ++kitem;
      }
      // After an abort some loads may have no consumer: wait (bounded) for the
      // last fill of every stage and of K/V so that no copy is in flight when
      // the CTA exits.
      ptx::CtaCtl no_abort{0, 0};
      if constexpr (kSt == 1) {  // the last fill of every atom (a step may have stopped half loaded)
        for (int a = 0; a < Lay::kAtoms; ++a) {
          if (nq_loads[a]) ptx::mbar_wait(q_full + a, (nq_loads[a] - 1) & 1, &no_abort, nullptr, kSiteBwdDrain, budget);
          if (ndo_loads[a])
            ptx::mbar_wait(do_full + a, (ndo_loads[a] - 1) & 1, &no_abort, nullptr, kSiteBwdDrain, budget);
        }
      } else {
        for (uint32_t q = pos > kSt ? pos - kSt : 0; q < pos; ++q) {
          ptx::mbar_wait(q_full + q % kSt, (q / kSt) & 1, &no_abort, nullptr, kSiteBwdDrain, budget);
          ptx::mbar_wait(do_full + q % kSt, (q / kSt) & 1, &no_abort, nullptr, kSiteBwdDrain, budget);
        }
      }
      if (kitem > 0) {  // the last fills of V and (if its wait was reached) K
        ptx::mbar_wait(v_full, (kitem - 1) & 1, &no_abort, nullptr, kSiteBwdDrain, budget);
        ptx::mbar_wait(k_full, (kitem - 1) & 1, &no_abort, nullptr, kSiteBwdDrain, budget);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (every value it computes is warp-uniform)
    // and one elected lane issues each group of MMAs and commits: a converged
    // warp issues at the tensor-core rate, a loop run by one lane does not.
    // Barriers that are usually complete long before (dO, the next Q, the
    // accumulators) are waited for ahead of the real dependency, so that their
    // shared-memory latency overlaps that wait instead of following it.
    uint32_t pos = 0, x = 0, kitem = 0;
    bool ok = true;
    const uint32_t k_addr = ptx::smem_u32(smem + Lay::kOffK);
    const uint32_t v_addr = ptx::smem_u32(smem + Lay::kOffV);
    const uint32_t ds_addr = ptx::smem_u32(smem + Lay::kOffDS);
    auto wait = [&](uint64_t* bar, uint32_t parity, int site) -> bool {
      return ptx::warp_all(ptx::mbar_wait(bar, parity, ctl, status, site, budget));
    };
    for (int v = blockIdx.x; ok && v < n_work; v += gridDim.x) {
      const BwdItem I = bwd_item(p, v);
      if (I.nq <= 0) continue;
      const int ca = slice_col<D, DC>(p, I) >> 6;  // first atom of the item's slice
      if (!(ok = wait(k_full, kitem & 1, kSiteBwdMmaKV))) break;
      ptx::tc_fence_after();
      if (lane == 0) tw.rec(trace::kBwd, trace::kBwdItem, kitem);
      // S^T(x) = K Q^T. With two Q/dO stages it is issued for the first query
      // tile of the item at the start of the tile and for every later one right
      // after dS^T of the previous tile, so the softmax of tile x + 1 overlaps
      // the dK / dQ MMAs of tile x; with one stage, at the start of its own tile.
      // Called by the elected lane.
      auto issue_s = [&](uint32_t stage) {
        const uint32_t qa = ptx::smem_u32(smem + Lay::kOffQ + stage * Lay::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          ptx::mma_ss(tmem + Lay::kColS, ptx::sdesc_sw128(k_addr + off, 16, 1024),
                      ptx::sdesc_sw128(qa + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(s_full);
      };
      auto wait_q = [&](uint32_t ps) -> bool { return wait(q_full + ps % kSt, (ps / kSt) & 1, kSiteBwdMmaQ); };
      // One stage: S^T (A = K, B = Q) or dP^T (A = V, B = dO) over the atoms of
      // Q or dO as they arrive, slice c last; the atoms outside the slice go
      // back to the producer when the product completes.
      auto atoms_mma = [&](uint32_t d_col, uint32_t a_addr, uint32_t b_addr, uint64_t* full, uint64_t* empty,
                           uint64_t* done) -> bool {
        for (int n = 0; n < Lay::kAtoms; ++n) {
          const int a = atom_at(n, ca, kSliceAtoms, Lay::kAtoms);
          if (!wait(full + a, x & 1, kSiteBwdMmaQ)) return false;
          ptx::tc_fence_after();
          if (ptx::elect_one()) {
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const uint32_t off = a * 16384 + k4 * 32;
              ptx::mma_ss(tmem + d_col, ptx::sdesc_sw128(a_addr + off, 16, 1024),
                          ptx::sdesc_sw128(b_addr + off, 16, 1024), kIdS, (n > 0 || k4 > 0) ? 1u : 0u);
            }
            if (n + 1 == Lay::kAtoms) {
              ptx::mma_commit(done);
              for (int m = 0; m < Lay::kAtoms - kSliceAtoms; ++m)
                ptx::mma_commit(empty + atom_at(m, ca, kSliceAtoms, Lay::kAtoms));
            }
          }
          __syncwarp();
        }
        return true;
      };
      for (int ii = 0; ii < I.nq; ++ii, ++x) {
        const uint32_t st = pos % kSt;
        const uint32_t q_addr = ptx::smem_u32(smem + Lay::kOffQ + st * Lay::kTileBytes);
        const uint32_t do_addr = ptx::smem_u32(smem + Lay::kOffDO + st * Lay::kTileBytes);
        if constexpr (kSt == 1) {
          if (lane == 0) tw.rec(trace::kBwd, trace::kBwdSIssue, x);
          if (!(ok = atoms_mma(Lay::kColS, k_addr, q_addr, q_full, q_empty, s_full))) break;
          // dP^T = V dO^T into the columns dQ of the previous tile used
          if (x > 0 && !(ok = wait(dq_free, (x - 1) & 1, kSiteBwdMmaDQFree))) break;
          if (ii == 0 && !(ok = wait(v_full, kitem & 1, kSiteBwdMmaKV))) break;
          if (lane == 0) tw.rec(trace::kBwd, trace::kBwdDPIssue, x);
          if (!(ok = atoms_mma(Lay::kColDP, v_addr, do_addr, do_full, do_empty, dp_full))) break;
          if (ii + 1 == I.nq) {  // the item's last dP^T was V's last reader
            if (ptx::elect_one()) ptx::mma_commit(v_empty);
            __syncwarp();
          }
        } else {
          if (ii == 0) {
            if (!(ok = wait_q(pos))) break;
            ptx::tc_fence_after();
            if (lane == 0) tw.rec(trace::kBwd, trace::kBwdSIssue, x);
            if (ptx::elect_one()) issue_s(st);
            __syncwarp();
          }
          // dP^T = V dO^T into the columns dQ of the previous tile used
          if (!(ok = wait(do_full + st, (pos / kSt) & 1, kSiteBwdMmaQ))) break;
          if (x > 0 && !(ok = wait(dq_free, (x - 1) & 1, kSiteBwdMmaDQFree))) break;
          if (ii == 0 && !(ok = wait(v_full, kitem & 1, kSiteBwdMmaKV))) break;
          ptx::tc_fence_after();
          if (lane == 0) tw.rec(trace::kBwd, trace::kBwdDPIssue, x);
          if (ptx::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              ptx::mma_ss(tmem + Lay::kColDP, ptx::sdesc_sw128(v_addr + off, 16, 1024),
                          ptx::sdesc_sw128(do_addr + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(dp_full);
            if (ii + 1 == I.nq) ptx::mma_commit(v_empty);  // the item's last dP^T was V's last reader
          }
          __syncwarp();
        }
        // dV += P^T dO[:, slice]
        if (ii == 0 && kitem > 0 && !(ok = wait(acc_free, (kitem - 1) & 1, kSiteBwdMmaAccFree))) break;
        if (!(ok = wait(p_full, x & 1, kSiteBwdMmaP))) break;
        ptx::tc_fence_after();
        if (lane == 0) tw.rec(trace::kBwd, trace::kBwdDVIssue, x);
        if (ptx::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            ptx::mma_ts(tmem + Lay::kColDV, tmem + Lay::kColS + 64 * (kk >> 2) + 8 * (kk & 3),
                        ptx::sdesc_sw128(do_addr + ca * 16384 + kk * 2048, 16384, 1024), kIdAcc,
                        (ii > 0 || kk > 0) ? 1u : 0u);
          }
          if constexpr (kSt == 1)  // dV was the last reader of the slice's dO atoms
            for (int k = 0; k < kSliceAtoms; ++k) ptx::mma_commit(do_empty + ca + k);
        }
        __syncwarp();
        const bool next_s = kSt > 1 && ii + 1 < I.nq;
        if (next_s && !(ok = wait_q(pos + 1))) break;
        if (!(ok = wait(ds_full, x & 1, kSiteBwdMmaDS))) break;
        ptx::tc_fence_after();
        if (lane == 0) {
          tw.rec(trace::kBwd, trace::kBwdDQDKIssue, x);
          if (next_s && kStageInDO) tw.rec(trace::kBwd, trace::kBwdSIssue, x + 1);  // issued between dQ and dK
        }
        if (ptx::elect_one()) {
          // dQ(tile) = dS K[:, slice] into the dP^T columns (the softmax has read dP^T)
          auto mma_dq = [&]() {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              ptx::mma_ss(tmem + Lay::kColDP, ptx::sdesc_sw128(ds_addr + kk * 2048, 16384, 1024),
                          ptx::sdesc_sw128(k_addr + ca * 16384 + kk * 2048, 16384, 1024), kIdDQ,
                          kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(dq_full);
          };
          // dK += dS^T Q[:, slice]: dS^T from the swizzled shared-memory copy
          // (K-major view), or with one stage from its TMEM copy (each group's
          // 64 query columns packed over the first 32 of its dP^T columns)
          auto mma_dk = [&]() {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              const uint64_t q_desc = ptx::sdesc_sw128(q_addr + ca * 16384 + kk * 2048, 16384, 1024);
              if (kStageInDO) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                ptx::mma_ss(tmem + Lay::kColDK, ptx::sdesc_sw128(ds_addr + off, 16, 1024), q_desc, kIdAcc,
                            (ii > 0 || kk > 0) ? 1u : 0u);
              } else {
                ptx::mma_ts(tmem + Lay::kColDK, tmem + Lay::kColDP + 64 * (kk >> 2) + 8 * (kk & 3), q_desc, kIdAcc,
                            (ii > 0 || kk > 0) ? 1u : 0u);
              }
            }
          };
          if (kStageInDO) {
            // dQ first, so that its drain (staged in this tile's dO buffer)
            // overlaps the next S^T and dK; the S^T columns are free once dV has
            // been issued and the softmax has read P^T back. dK is the last
            // reader of Q (the softmax read the rows before dS^T); the last
            // tile's stage is released by the epilogue, which stages dK and dV
            // there.
            mma_dq();
            if (ii + 1 == I.nq) ptx::mma_commit(k_empty);  // the item's last dQ was K's last reader
            if (next_s) issue_s((pos + 1) % kSt);
            mma_dk();
            if (ii + 1 < I.nq) ptx::mma_commit(q_empty + st);
          } else {
            // one stage: dQ is staged in the dS buffer, so dK reads dS first;
            // Q atom c (read by dK) and the LSE / delta rows go back to the
            // producer before dQ, as the next tile's S^T waits for them
            mma_dk();
            for (int k = 0; k < kSliceAtoms; ++k) ptx::mma_commit(q_empty + ca + k);
            mma_dq();
            if (ii + 1 == I.nq) ptx::mma_commit(k_empty);  // the item's last dQ was K's last reader
          }
          ptx::mma_commit(ds_free);  // dQ and dK have read dS
        }
        __syncwarp();
        ++pos;
      }
      if (!ok) break;
      if (ptx::elect_one()) ptx::mma_commit(acc_full);
      __syncwarp();
      ++kitem;
    }
    if (ptx::elect_one()) ptx::mma_commit(drain);
    __syncwarp();
    ptx::CtaCtl no_abort{0, 0};
    ptx::mbar_wait(drain, 0, &no_abort, nullptr, kSiteBwdDrain, budget);
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ P^T and dS^T (thread = key row)
    // group g = warp / 4 takes query columns 64 g .. 64 g + 63
    const int g = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_cols = tmem + lane_base + Lay::kColS + 64 * g;    // S^T, then packed P^T
    const uint32_t dp_cols = tmem + lane_base + Lay::kColDP + 64 * g;  // dP^T, then packed dS^T
    const float sl = p.scale_log2;
    const uint64_t sl2 = ptx::f2_packf(sl, sl);
    uint32_t pos = 0, x = 0;
    bool ok = true;
    uint8_t* ds_row = smem + Lay::kOffDS + g * 16384 + r * 128;  // this group's atom of dS
    const int sw = r & 7;
    for (int v = blockIdx.x; ok && v < n_work; v += gridDim.x) {
      const BwdItem I = bwd_item(p, v);
      if (I.nq <= 0) continue;
      const int rk = I.Lk - kTile * I.t;  // valid key rows of the tile
      for (int ii = 0; ii < I.nq; ++ii, ++x) {
        int g_unused, i;
        bwd_step(I, ii, g_unused, i);
        const uint32_t st = pos % kSt;
        const float* lse2 = reinterpret_cast<const float*>(smem + Lay::kOffRow + st * 1024) + 64 * g;
        const float* dlt = lse2 + 128;
        const int rq = I.Lq - kTile * i;  // valid query columns
        // tiles that cross the (bottom-right aligned) diagonal or the end of a sequence
        const bool masked = rk < kTile || rq < kTile || (p.causal && kTile * I.t + kTile - 1 > kTile * i + I.delta);
        // visible query columns c of this key row: c_lo <= c < c_hi (causal: query
        // 128 i + c sees key 128 t + r iff 128 i + c >= 128 t + r - delta)
        const int c_lo = p.causal ? max(0, kTile * (I.t - i) + r - I.delta) : 0;
        const int c_hi = r < rk ? rq : 0;
        if (!(ok = ptx::mbar_wait(s_full, x & 1, ctl, status, kSiteBwdSoftS, budget))) break;
        ptx::tc_fence_after();
        if (lane == 0) tw.rec(trace::kBwd, trace::kBwdPBegin, x);
        // P^T = 2^(S^T * scale * log2e - lse2[q]), two chunks of 32 query columns
        {
          uint32_t sv[2][32];
          ptx::tmem_ld32(s_cols, sv[0]);
          ptx::tmem_ld32(s_cols + 32, sv[1]);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(sv[0]);
          ptx::reg_fence32(sv[1]);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint32_t pk[16];
            const int cb = 64 * g + 32 * u;  // first query column of the chunk
            float lq[32];  // -lse2 of the 32 query columns (same for every lane: broadcast reads)
#pragma unroll
            for (int e = 0; e < 8; ++e)
              *reinterpret_cast<float4*>(lq + 4 * e) = reinterpret_cast<const float4*>(lse2 + 32 * u)[e];
            // branch-free; the masked form only on edge tiles (with the tensor
            // core reading shared memory, extra instructions here cost a lot)
            if (!masked) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float x0, x1;
                ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(sv[u][2 * e], sv[u][2 * e + 1]), sl2,
                                           ptx::f2_packf(lq[2 * e], lq[2 * e + 1])),
                               x0, x1);
                pk[e] = ptx::pack_bf16(ptx::ex2(x0), ptx::ex2(x1));
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int c0 = cb + 2 * e;
                float x0, x1;
                ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(sv[u][2 * e], sv[u][2 * e + 1]), sl2,
                                           ptx::f2_packf(lq[2 * e], lq[2 * e + 1])),
                               x0, x1);
                float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                p0 = (c0 >= c_lo && c0 < c_hi) ? p0 : 0.f;
                p1 = (c0 + 1 >= c_lo && c0 + 1 < c_hi) ? p1 : 0.f;
                pk[e] = ptx::pack_bf16(p0, p1);
              }
            }
            ptx::tmem_st16(s_cols + 16 * u, pk);  // over S^T columns this thread has read
          }
        }
        // dP^T and the dS buffer, tested while the P^T stores drain
        const bool dp_ready = ptx::mbar_test(dp_full, x & 1);
        const bool ds_ready = x == 0 || ptx::mbar_test(ds_free, (x - 1) & 1);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full);
        if (lane == 0) tw.rec(trace::kBwd, trace::kBwdPEnd, x);
        // dS^T = P^T * (dP^T - delta[q])
        if (!dp_ready && !(ok = ptx::mbar_wait(dp_full, x & 1, ctl, status, kSiteBwdSoftDP, budget))) break;
        ptx::tc_fence_after();
        if (x > 0) {  // the MMAs of the previous tile have read dS (and TMA the dQ staged there)
          if (!ds_ready && !(ok = ptx::mbar_wait(ds_free, (x - 1) & 1, ctl, status, kSiteBwdSoftDP, budget))) break;
          if (!kStageInDO && !(ok = ptx::mbar_wait(stage_free, (x - 1) & 1, ctl, status, kSiteBwdSoftDP, budget)))
            break;
        }
        if (lane == 0) tw.rec(trace::kBwd, trace::kBwdDSBegin, x);
#pragma unroll 1
        for (int k = 0; k < 2; ++k) {  // two chunks of 32 query columns
          uint32_t dp[32];
          uint32_t pp[16];
          uint32_t dsw[16];  // dS^T for the TMEM copy (one stage only)
          ptx::tmem_ld32(dp_cols + 32 * k, dp);
          ptx::tmem_ld16(s_cols + 16 * k, pp);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(dp);
#pragma unroll
          for (int e = 0; e < 16; ++e) asm volatile("" : "+r"(pp[e]));
          // 32 query columns = half of a 128-byte swizzled row of this group's atom
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int ch = 4 * k + c4;  // 16-byte chunk of the atom row
            uint32_t w[4];
            float dq8[8];  // -delta of the 8 query columns (broadcast reads)
            *reinterpret_cast<float4*>(dq8) = reinterpret_cast<const float4*>(dlt + 8 * ch)[0];
            *reinterpret_cast<float4*>(dq8 + 4) = reinterpret_cast<const float4*>(dlt + 8 * ch)[1];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int cl = 8 * c4 + 2 * e;  // column within the 32-wide chunk (even)
              const uint32_t pw = pp[cl / 2];
              // (dP - delta) and P (bf16 pair widened) multiplied on fp32 pairs
              const uint64_t d2 = ptx::f2_add(ptx::f2_pack(dp[cl], dp[cl + 1]), ptx::f2_packf(dq8[2 * e], dq8[2 * e + 1]));
              float s0, s1;
              ptx::f2_unpack(ptx::f2_mul(ptx::f2_packf(ptx::bf16lo(pw), ptx::bf16hi(pw)), d2), s0, s1);
              w[e] = ptx::pack_bf16(s0, s1);
              if constexpr (!kStageInDO) dsw[4 * c4 + e] = w[e];
            }
            uint4* dst = reinterpret_cast<uint4*>(ds_row + ((ch ^ sw) << 4));
            *dst = make_uint4(w[0], w[1], w[2], w[3]);
          }
          // one stage: dS^T of these 32 query columns, two bf16 per column, over
          // dP^T columns this thread has read (the A operand of dK from TMEM)
          if constexpr (!kStageInDO) ptx::tmem_st16(dp_cols + 16 * k, dsw);
        }
        if constexpr (!kStageInDO) ptx::tmem_st_wait();
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ds_full);
        if (lane == 0) tw.rec(trace::kBwd, trace::kBwdDSEnd, x);
        ++pos;
      }
    }
  } else if (warp >= 10) {
    // ------------------------------------------------------------ dQ drain + dK/dV epilogue (warps 10-13)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t x = 0, kitem = 0, ns = 0, nr = 0;  // rounds of dQ staged; waits on stage_read
    bool ok = true;
    for (int v = blockIdx.x; ok && v < n_work; v += gridDim.x) {
      const BwdItem I = bwd_item(p, v);
      if (I.nq <= 0) {
        // a varlen key tile that no query sees: its dK and dV rows are zero
        if (p.var) {
          const int64_t orow = (static_cast<int64_t>(I.kv_row0 + r) * p.kv_heads + I.h) * D + slice_col<D, DC>(p, I);
          if (r < I.Lk - kTile * I.t)
            for (int c8 = 0; c8 < DC; c8 += 8) {
              ptx::st_v4(p.dv + orow + c8, 0, 0, 0, 0);
              ptx::st_v4(p.dk + orow + c8, 0, 0, 0, 0);
            }
        }
        continue;
      }
      for (int ii = 0; ii < I.nq; ++ii, ++x) {
        int g, i;
        bwd_step(I, ii, g, i);
        if (!(ok = ptx::mbar_wait(dq_full, x & 1, ctl, status, kSiteBwdDQ, budget))) break;
        ptx::tc_fence_after();
        if (lane == 0) tw.rec(trace::kBwd, trace::kBwdDQBegin, x);
        // dQ leaves TMEM a staging round (a buffer-full of 32-column fp32 boxes,
        // 16 KB each, 128B swizzle) at a time: in this tile's dO stage buffer
        // with two stages (then released to the producer), in the dS buffer
        // with one (then the softmax may write the next dS). The dQ columns are
        // released as soon as the last round is in registers (the next dP^T
        // goes there); TMA adds each round into the accumulator. Rows past the
        // sequence hold exact zeros (their dS is masked), so whole boxes are added.
        const int qrow = I.q_row0 + kTile * i;
        const int xcol = (I.hq0 + g) * D + slice_col<D, DC>(p, I);  // dQ of query head hq0 + g
        const bool issuer = warp == 10 && lane == 0;
        const uint32_t st = x % kSt;
        uint8_t* stage = kStageInDO ? smem + Lay::kOffDO + st * Lay::kTileBytes : smem + Lay::kOffDS;
        constexpr int kBoxesPerRound = kStageInDO ? Lay::kTileBytes / 16384 : 2;
        constexpr int kRounds = (DC / 32) / kBoxesPerRound;
        constexpr int kRoundCols = 32 * kBoxesPerRound;
        static_assert(kRounds == 1 || kRounds == 2, "dQ staging rounds");
        uint32_t dq[kRoundCols];
        auto tmem_read = [&](int rd) {
#pragma unroll
          for (int c = 0; c < kRoundCols / 32; ++c)
            ptx::tmem_ld32(tmem + lane_base + Lay::kColDP + kRoundCols * rd + 32 * c,
                           *reinterpret_cast<uint32_t(*)[32]>(dq + 32 * c));
          ptx::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kRoundCols / 32; ++c) ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(dq + 32 * c));
        };
        auto release_dq = [&]() {  // all of dQ is out of TMEM: the next dP^T may go there
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(dq_free);
        };
        auto write_round = [&]() {
#pragma unroll
          for (int b = 0; b < kBoxesPerRound; ++b) {
            uint8_t* row = stage + b * 16384 + r * 128;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int k = 32 * b + 4 * e;
              ptx::st_shared_v4(row + ((e ^ (r & 7)) << 4), dq[k], dq[k + 1], dq[k + 2], dq[k + 3]);
            }
          }
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive(staged);
        };
        // Every drain thread waits for a whole round before the next: a thread
        // that ran on must not arrive on `staged` again before this phase has
        // completed, or the phase would complete without the writes of a slower
        // thread. The issuer then hands the round to TMA.
        auto finish_round = [&](int rd) -> bool {
          if (!ptx::mbar_wait(staged, ns & 1, ctl, status, kSiteBwdDQ, budget)) return false;
          if (issuer) {
#pragma unroll
            for (int b = 0; b < kBoxesPerRound; ++b)
              ptx::tma_reduce_add_2d(&tm_dq, stage + b * 16384, xcol + kRoundCols * rd + 32 * b, qrow);
            ptx::bulk_commit();
          }
          ++ns;
          return true;
        };
        // round 0 goes to shared memory before round 1 leaves TMEM, so the dQ
        // columns are released without waiting for any TMA read
        tmem_read(0);
        write_round();
        if (kRounds == 2) tmem_read(1);
        release_dq();
        if (!(ok = finish_round(0))) break;
        if (kRounds == 2) {
          if (issuer) {  // the reduce-adds of round 0 have read the staging
            ptx::bulk_wait_read0();
            ptx::mbar_arrive(stage_read);
          }
          if (!(ok = ptx::mbar_wait(stage_read, nr & 1, ctl, status, kSiteBwdDQ, budget))) break;
          ++nr;
          write_round();
          if (!(ok = finish_round(1))) break;
        }
        if (issuer) ptx::bulk_wait_read0();
        if (!ok) break;
        if (lane == 0) tw.rec(trace::kBwd, trace::kBwdDQEnd, x);
        if (issuer && !(kStageInDO && ii + 1 == I.nq)) ptx::mbar_arrive(kStageInDO ? do_empty + st : stage_free);
      }
      if (!ok) break;
      if (!(ok = ptx::mbar_wait(acc_full, kitem & 1, ctl, status, kSiteBwdEpi, budget))) break;
      ptx::tc_fence_after();
      if (lane == 0) tw.rec(trace::kBwd, trace::kBwdAccBegin, kitem);
      const bool issuer = warp == 10 && lane == 0;
      const uint32_t st_last = (x - 1) % kSt;  // stage of the item's last query tile
      const bool full_tile = I.Lk - kTile * I.t >= kTile;
      auto release_acc = [&]() {  // dV and dK are out of TMEM: the next item may accumulate
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(acc_free);
      };
      if (kStageInDO && full_tile) {
        // dV and dK go to global memory by TMA: staged as bf16 (128B swizzle,
        // 64-column atoms) in the Q and dO buffers of the last tile's stage,
        // which the producer gets back once the stores have read them.
        uint8_t* sv = smem + Lay::kOffQ + st_last * Lay::kTileBytes;
        uint8_t* sk = smem + Lay::kOffDO + st_last * Lay::kTileBytes;
        // the last tile's dQ reduce-adds have read their staging in the dO buffer
        if (issuer) {
          ptx::bulk_wait_read0();
          ptx::mbar_arrive(stage_read);
        }
        if (!(ok = ptx::mbar_wait(stage_read, nr & 1, ctl, status, kSiteBwdEpi, budget))) break;
        ++nr;
#pragma unroll 1
        for (int c = 0; c < DC / 32; ++c) {
          uint32_t a[32], b[32];
          ptx::tmem_ld32(tmem + lane_base + Lay::kColDV + 32 * c, a);
          ptx::tmem_ld32(tmem + lane_base + Lay::kColDK + 32 * c, b);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(a);
          ptx::reg_fence32(b);
          if (c == DC / 32 - 1) release_acc();
          const int off = (c >> 1) * 16384 + r * 128;  // atom of these 32 columns, this row
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t wv[4], wk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              wv[e] = ptx::pack_bf16(__uint_as_float(a[8 * q4 + 2 * e]), __uint_as_float(a[8 * q4 + 2 * e + 1]));
              wk[e] = ptx::pack_bf16(__uint_as_float(b[8 * q4 + 2 * e]) * p.scale,
                                     __uint_as_float(b[8 * q4 + 2 * e + 1]) * p.scale);
            }
            const int chunk = ((((c & 1) << 2) + q4) ^ (r & 7)) << 4;
            ptx::st_shared_v4(sv + off + chunk, wv[0], wv[1], wv[2], wv[3]);
            ptx::st_shared_v4(sk + off + chunk, wk[0], wk[1], wk[2], wk[3]);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(staged);
        if (!(ok = ptx::mbar_wait(staged, ns & 1, ctl, status, kSiteBwdEpi, budget))) break;
        ++ns;
        if (issuer) {
          const int xcol = I.h * D + slice_col<D, DC>(p, I);
#pragma unroll
          for (int at = 0; at < DC / 64; ++at) {
            ptx::tma_store_2d(&tm_dv, sv + at * 16384, xcol + 64 * at, I.kv_row0);
            ptx::tma_store_2d(&tm_dk, sk + at * 16384, xcol + 64 * at, I.kv_row0);
          }
          ptx::bulk_commit();
          ptx::bulk_wait_read0();
          ptx::mbar_arrive(q_empty + st_last);
          ptx::mbar_arrive(do_empty + st_last);
        }
      } else {
        // a partial key tile (its rows end inside the 128-row box) or a single
        // stage: every thread stores its own row
        const bool k_ok = r < I.Lk - kTile * I.t;
        const int64_t orow = (static_cast<int64_t>(I.kv_row0 + r) * p.kv_heads + I.h) * D + slice_col<D, DC>(p, I);
#pragma unroll 1
        for (int c = 0; c < DC / 32; ++c) {
          uint32_t a[32], b[32];
          ptx::tmem_ld32(tmem + lane_base + Lay::kColDV + 32 * c, a);
          ptx::tmem_ld32(tmem + lane_base + Lay::kColDK + 32 * c, b);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(a);
          ptx::reg_fence32(b);
          if (c == DC / 32 - 1) release_acc();
          if (k_ok) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t wv[4], wk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                wv[e] = ptx::pack_bf16(__uint_as_float(a[8 * q4 + 2 * e]), __uint_as_float(a[8 * q4 + 2 * e + 1]));
                wk[e] = ptx::pack_bf16(__uint_as_float(b[8 * q4 + 2 * e]) * p.scale,
                                       __uint_as_float(b[8 * q4 + 2 * e + 1]) * p.scale);
              }
              ptx::st_v4(p.dv + orow + 32 * c + 8 * q4, wv[0], wv[1], wv[2], wv[3]);
              ptx::st_v4(p.dk + orow + 32 * c + 8 * q4, wk[0], wk[1], wk[2], wk[3]);
            }
          }
        }
        if (kStageInDO && issuer) {  // the last tile's stage: Q was read by dK, dO by dV and the dQ staging
          ptx::mbar_arrive(q_empty + st_last);
          ptx::mbar_arrive(do_empty + st_last);
        }
      }
      if (lane == 0) tw.rec(trace::kBwd, trace::kBwdAccEnd, kitem);
      ++kitem;
    }
    if (warp == 10 && lane == 0) ptx::bulk_wait0();  // every reduce-add has completed
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

// ------------------------------------------------------------------ pre / post

// delta = rowsum(dO * O) and lse2 = LSE * log2(e), both stored negated (the
// backward adds them with paired fp32 instructions), written in a layout padded
// to whole 128-row query tiles (zeros past the end of a sequence), so that the
// backward can fetch one tile's 128 values with a single aligned bulk copy.
// The same pass zeroes the tile's rows of the fp32 dQ accumulator (broadcast-Q:
// the shared Q's rows, once, by the CTAs of sequence 0).
// One CTA per padded query tile (blockIdx.x) and head (blockIdx.y). A row's
// d elements are read 16 bytes per lane by a group of kRowLanes lanes, a warp
// takes 32 / kRowLanes rows at a time, and every load of a warp's 16 rows is
// issued before the first sum, so that 64 KB of a tile are in flight at once.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      const float* __restrict__ lse, const int32_t* offsets,
                                                      const int32_t* tile_base, const int32_t* status, int batch,
                                                      int heads, int total, int bcast, int q_len, int pad_tiles,
                                                      float* __restrict__ lse2p, float* __restrict__ deltap,
                                                      float* __restrict__ dq_acc) {
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr int kChunks = D / 8;                                             // 16-byte chunks of a row
  constexpr int kRowLanes = kChunks <= 8 ? 8 : (kChunks <= 16 ? 16 : 32);   // lanes per row (power of two)
  constexpr int kRowsPerWarp = 32 / kRowLanes;
  constexpr int kIters = (kTile / 8) / kRowsPerWarp;  // rows of a warp / rows per pass
  wait_prior_grid();
  allow_next_grid();
  const int gt = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (status[0] != JFA_OK) return;
  // locate the tile: self -> (b, i) by binary search over tile_base; broadcast -> (b, i) directly
  int b, i, Lq;
  int64_t qrow0, lse_base, pad_base, acc_row0;
  if (!bcast) {
    if (gt >= tile_base[batch]) return;
    int lo = 0, hi = batch;  // largest b with tile_base[b] <= gt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tile_base[mid] <= gt) lo = mid; else hi = mid;
    }
    b = lo;
    while (b + 1 < batch && tile_base[b + 1] <= gt) ++b;
    i = gt - tile_base[b];
    const int s0 = offsets[b];
    Lq = offsets[b + 1] - s0;
    qrow0 = s0 + static_cast<int64_t>(kTile) * i;
    lse_base = static_cast<int64_t>(h) * total + qrow0;
    pad_base = (static_cast<int64_t>(h) * pad_tiles + gt) * kTile;
    acc_row0 = qrow0;
  } else {
    const int nqt = (q_len + kTile - 1) / kTile;
    b = gt / nqt;
    i = gt - b * nqt;
    if (b >= batch) return;
    Lq = q_len;
    qrow0 = static_cast<int64_t>(b) * q_len + static_cast<int64_t>(kTile) * i;
    lse_base = (static_cast<int64_t>(b) * heads + h) * q_len + static_cast<int64_t>(kTile) * i;
    pad_base = ((static_cast<int64_t>(b) * heads + h) * nqt + i) * kTile;
    acc_row0 = b == 0 ? static_cast<int64_t>(kTile) * i : -1;  // the shared Q's rows, zeroed once
  }
  const int sub = lane / kRowLanes, cl = lane % kRowLanes;  // row within the pass, chunk lane
  const int rows_valid = min(kTile, Lq - kTile * i);
  constexpr int kBatch = kIters > 8 ? 8 : kIters;  // passes whose loads are in flight together
#pragma unroll
  for (int i0 = 0; i0 < kIters; i0 += kBatch) {
    uint4 a[kBatch], c[kBatch];
#pragma unroll
    for (int it = 0; it < kBatch; ++it) {
      const int r = warp * (kTile / 8) + (i0 + it) * kRowsPerWarp + sub;
      a[it] = make_uint4(0, 0, 0, 0);
      c[it] = make_uint4(0, 0, 0, 0);
      if (r < rows_valid && cl < kChunks) {
        const int64_t off = ((qrow0 + r) * heads + h) * D + 8 * cl;
        a[it] = ptx::ld_nc_v4(o + off);
        c[it] = ptx::ld_nc_v4(dout + off);
      }
    }
#pragma unroll
    for (int it = 0; it < kBatch; ++it) {
      const int r = warp * (kTile / 8) + (i0 + it) * kRowsPerWarp + sub;
      const uint32_t* av = reinterpret_cast<const uint32_t*>(&a[it]);
      const uint32_t* cv = reinterpret_cast<const uint32_t*>(&c[it]);
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(ptx::bf16lo(av[e]), ptx::bf16lo(cv[e]), acc);
        acc = fmaf(ptx::bf16hi(av[e]), ptx::bf16hi(cv[e]), acc);
      }
#pragma unroll
      for (int off = kRowLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (cl == 0) {
        const bool ok = r < rows_valid;
        deltap[pad_base + r] = ok ? -acc : 0.f;
        lse2p[pad_base + r] = ok ? -lse[lse_base + r] * kLog2e : 0.f;
      }
    }
  }
  // zero this tile's rows of the dQ accumulator: one 16-byte store per thread per step
  if (acc_row0 >= 0) {
    constexpr int kRowStores = D / 4;  // float4 per row
    for (int k = threadIdx.x; k < rows_valid * kRowStores; k += blockDim.x) {
      const int r = k / kRowStores, e = k - r * kRowStores;
      reinterpret_cast<float4*>(dq_acc + ((acc_row0 + r) * heads + h) * D)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// dQ = scale * dQ_accumulated, fp32 -> bf16, four elements per thread.
__global__ void bwd_post_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq, int64_t n4, float scale,
                                const int32_t* status) {
  wait_prior_grid();
  if (status[0] != JFA_OK) return;
  for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n4;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = acc[k];
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x * scale, v.y * scale);
    __nv_bfloat162 c = __floats2bfloat162_rn(v.z * scale, v.w * scale);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&a);
    w.y = *reinterpret_cast<uint32_t*>(&c);
    dq[k] = w;
  }
}

// ------------------------------------------------------------------ launchers

template <int D, int DC>
static cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                                const CUtensorMap& tdv, const BwdParams& p, int grid,
                                cudaStream_t stream) {
  using Lay = BwdLayout<D, DC>;
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(bwd_kernel<D, DC>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kAlloc);
  });
  if (e != cudaSuccess) return e;
  return launch_after(bwd_kernel<D, DC>, dim3(grid), dim3(448), Lay::kAlloc, stream, tq, tk, tv, tdo, tdq, tdk, tdv, p);
}

cudaError_t launch_bwd_main(const BwdLaunch& L, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, cudaStream_t stream) {
  BwdParams p;
  p.offsets = L.offsets;
  p.tile_base = L.tile_base;
  p.item_seq = L.item_seq;
  p.items = L.items;
  p.status = L.status;
  p.lse2p = L.lse2p;
  p.deltap = L.deltap;
  p.dk = static_cast<__nv_bfloat16*>(L.dk);
  p.dv = static_cast<__nv_bfloat16*>(L.dv);
  p.heads = L.heads;
  p.var = L.var;
  p.group = L.var ? L.group : 1;
  p.kv_heads = L.var ? L.kv_heads : L.heads;
  p.total = L.total;
  p.bcast = L.bcast;
  p.q_len = L.q_len;
  p.causal = L.causal;
  p.n_chunks = L.n_chunks > 0 ? L.n_chunks : L.head_dim / L.head_chunk;
  p.col0 = L.col0;
  p.chunk = L.head_chunk;
  p.pad_tiles = L.pad_tiles;
  p.scale = L.scale;
  p.scale_log2 = L.scale * 1.4426950408889634f;
  p.budget_ns = L.budget_ns;
  if (L.head_dim == 64 && L.head_chunk == 64) return launch_bwd_t<64, 64>(tq, tk, tv, tdo, tdq, tdk, tdv, p, L.grid, stream);
  if (L.head_dim == 128 && L.head_chunk == 128) return launch_bwd_t<128, 128>(tq, tk, tv, tdo, tdq, tdk, tdv, p, L.grid, stream);
  if (L.head_dim == 128 && L.head_chunk == 64) return launch_bwd_t<128, 64>(tq, tk, tv, tdo, tdq, tdk, tdv, p, L.grid, stream);
  if (L.head_dim == 192 && L.head_chunk == 64) return launch_bwd_t<192, 64>(tq, tk, tv, tdo, tdq, tdk, tdv, p, L.grid, stream);
  if (L.head_dim == 192 && L.head_chunk == 128) return launch_bwd_t<192, 128>(tq, tk, tv, tdo, tdq, tdk, tdv, p, L.grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_pre(int head_dim, const void* o, const void* dout, const float* lse, const int32_t* offsets,
                           const int32_t* tile_base, const int32_t* status, int batch, int heads, int total, int bcast,
                           int q_len, int pad_tiles, int grid_tiles, float* lse2p, float* deltap, float* dq_acc,
                           cudaStream_t stream) {
  dim3 grid(grid_tiles, heads);
  auto O = static_cast<const __nv_bfloat16*>(o);
  auto dO = static_cast<const __nv_bfloat16*>(dout);
  cudaError_t e;
  if (head_dim == 64)
    e = launch_after(bwd_pre_kernel<64>, grid, dim3(256), 0, stream, O, dO, lse, offsets, tile_base, status, batch,
                     heads, total, bcast, q_len, pad_tiles, lse2p, deltap, dq_acc);
  else if (head_dim == 128)
    e = launch_after(bwd_pre_kernel<128>, grid, dim3(256), 0, stream, O, dO, lse, offsets, tile_base, status, batch,
                     heads, total, bcast, q_len, pad_tiles, lse2p, deltap, dq_acc);
  else if (head_dim == 192)
    e = launch_after(bwd_pre_kernel<192>, grid, dim3(256), 0, stream, O, dO, lse, offsets, tile_base, status, batch,
                     heads, total, bcast, q_len, pad_tiles, lse2p, deltap, dq_acc);
  else
    return cudaErrorInvalidValue;
  return e;
}

cudaError_t launch_bwd_post(const float* acc, void* dq, int64_t n, float scale, const int32_t* status, int sms,
                            cudaStream_t stream) {
  const int64_t n4 = n / 4;
  int64_t blocks = (n4 + 255) / 256;
  if (blocks > static_cast<int64_t>(sms) * 16) blocks = static_cast<int64_t>(sms) * 16;
  if (blocks < 1) blocks = 1;
  return launch_after(bwd_post_kernel, dim3(static_cast<int>(blocks)), dim3(256), 0, stream,
                      reinterpret_cast<const float4*>(acc), static_cast<uint2*>(dq), n4, scale, status);
}

}  // namespace jfa
