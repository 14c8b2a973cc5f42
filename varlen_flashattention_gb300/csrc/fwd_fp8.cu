// Jagged FlashAttention forward with FP8 (e4m3) inputs, head_dim 128.
//
// "Optimizing FlashAttention-4 for Efficient Inference" (hpjadul), section
// "PR 2109: Support FP8 Inputs": the inference forward takes FP8 inputs, for
// less memory traffic and faster tensor-core math than bf16. The page gives
// no scale convention; here each of Q, K, V carries one descale factor (a
// byte x stands for e4m3(x) * descale), O is bf16 and LSE fp32, as in jfa_fwd.
//
// Same pipeline as the per-tile forward (fwd.cu): a persistent grid walks the
// longest-first queue of (sequence, head, query tile) items; warp 4 loads
// tiles by TMA, warp 5 issues the MMAs, warps 0-3 run the online softmax
// (thread = query row) and the epilogue. What changes with 8-bit inputs:
//  * S = Q K^T and O += P V are tcgen05 MMAs of kind::f8f6f4 (K = 32 per
//    instruction); a 128 x 128 tile is 16 KB and one 128-byte swizzle row
//    holds a whole 128-element row, so Q, K and P stay K-major exactly as the
//    bf16 tiles do;
//  * O += P V needs V with the keys contiguous (the K-major B operand). A
//    pre-pass writes every 128-key tile of V transposed into its own
//    [head_dim x 128 keys] block (keys past the sequence zeroed), so each
//    block starts at x = 0 and every TMA start is 16-byte aligned;
//  * P (e4m3) goes to shared memory in the 128B-swizzled layout instead of
//    TMEM; its two buffers follow the two score buffers (the MMA that reads
//    P(x) completes before S(x + 2) is issued, and the softmax waits for
//    S(x + 2) before writing P(x + 2) into the same buffer);
//  * scores are scaled by scale * q_descale * k_descale; O by v_descale / l.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "jfa_internal.h"
#include "ptx.cuh"

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
  static constexpr int kSlots = 8;
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = kF8TileBytes;
  static constexpr int kOffP = kOffSlots + kSlots * kF8TileBytes;  // two P buffers
  static constexpr int kOffBars = kOffP + 2 * kF8TileBytes;
  // q_full, q_empty, slot_full[S], slot_empty[S], s_full[2], p_full[2], o_ready[2], o_free, drain
  static constexpr int kNumBars = 2 + 2 * kSlots + 2 + 2 + 2 + 1 + 1;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kTmemCols = 512;
  static_assert(kAlloc <= 232448, "shared memory budget");
};

struct Fp8Item {
  int h, t;
  int q_row, kv_row0, L, n_kv, vt0;
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
  return I;
}

template <bool CAUSAL>
__global__ void __launch_bounds__(192, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_vt, const Fp8Params p) {
  using Lay = Fp8Layout;
  constexpr int kSlots = Lay::kSlots;
  constexpr uint32_t kIdesc = idesc_e4m3(128, 128);

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
    ctl->abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_vt);
  }
  __syncthreads();
  if (warp == 5) {
    ptx::tmem_alloc(tmem_slot, Lay::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_items = p.status[2];
  int32_t* status = p.status;
  const uint64_t budget = p.budget_ns;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t pos = 0, kq = 0;
      bool ok = true;
      auto load_tile = [&](const CUtensorMap* map, int x, int y) -> bool {
        const uint32_t slot = pos % kSlots, round = pos / kSlots;
        if (!ptx::mbar_wait(slot_empty + slot, (round & 1) ^ 1, ctl, status, kSiteFwdProdSlot, budget)) return false;
        ptx::mbar_arrive_expect_tx(slot_full + slot, kF8TileBytes);
        ptx::tma_load_2d(smem + Lay::kOffSlots + slot * kF8TileBytes, map, slot_full + slot, x, y);
        ++pos;
        return true;
      };
      for (int idx = blockIdx.x; ok && idx < n_items; idx += gridDim.x) {
        const Fp8Item I = fp8_item(p, idx);
        if (I.n_kv == 0) continue;
        if (!ptx::mbar_wait(q_empty, (kq & 1) ^ 1, ctl, status, kSiteFwdProdQ, budget)) break;
        ptx::mbar_arrive_expect_tx(q_full, kF8TileBytes);
        ptx::tma_load_2d(smem + Lay::kOffQ, &tm_q, q_full, I.h * kF8D, I.q_row);
        // K_0, K_1, V_0, K_2, V_1, ...: V tile j is the transposed block vt0 + j of this head
        ok = load_tile(&tm_k, I.h * kF8D, I.kv_row0);
        for (int j = 0; ok && j < I.n_kv; ++j) {
          if (j + 1 < I.n_kv) ok = load_tile(&tm_k, I.h * kF8D, I.kv_row0 + kTile * (j + 1));
          if (ok) ok = load_tile(&tm_vt, 0, ((I.vt0 + j) * p.heads + I.h) * kF8D);
        }
        ++kq;
      }
      // an aborted pipeline may leave fills without a consumer: wait (bounded) for them
      ptx::CtaCtl no_abort{0, 0};
      for (uint32_t i = pos > kSlots ? pos - kSlots : 0; i < pos; ++i)
        ptx::mbar_wait(slot_full + i % kSlots, (i / kSlots) & 1, &no_abort, nullptr, kSiteFwdDrain, budget);
      if (kq > 0) ptx::mbar_wait(q_full, (kq - 1) & 1, &no_abort, nullptr, kSiteFwdDrain, budget);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t pos = 0, kq = 0, it = 0;
      const uint32_t q_addr = ptx::smem_u32(smem + Lay::kOffQ);
      bool ok = true;
      auto slot_wait = [&](uint32_t& slot) -> bool {
        slot = pos % kSlots;
        if (!ptx::mbar_wait(slot_full + slot, (pos / kSlots) & 1, ctl, status, kSiteFwdMmaSlot, budget)) return false;
        ptx::tc_fence_after();
        return true;
      };
      auto issue_qk = [&](uint32_t slot, uint32_t x) {  // S(x) = Q K^T, 4 x (K = 32)
        const uint32_t k_addr = ptx::smem_u32(smem + Lay::kOffSlots + slot * kF8TileBytes);
        const uint32_t d_tmem = tmem + ((x & 1) ? Lay::kColS1 : Lay::kColS0);
#pragma unroll
        for (int kk = 0; kk < kF8D / 32; ++kk)
          mma_ss_f8(d_tmem, ptx::sdesc_sw128(q_addr + kk * 32, 16, 1024),
                         ptx::sdesc_sw128(k_addr + kk * 32, 16, 1024), kIdesc, kk > 0 ? 1u : 0u);
        ptx::mma_commit(s_full + (x & 1));
        ptx::mma_commit(slot_empty + slot);
        ++pos;
      };
      for (int idx = blockIdx.x; ok && idx < n_items; idx += gridDim.x) {
        const Fp8Item I = fp8_item(p, idx);
        const int n = I.n_kv;
        if (n == 0) continue;
        if (!(ok = ptx::mbar_wait(q_full, kq & 1, ctl, status, kSiteFwdMmaQ, budget))) break;
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
          // O += P V: A = P (x & 1) in shared memory, B = the V^T block, both K-major over keys
          const uint32_t vt_addr = ptx::smem_u32(smem + Lay::kOffSlots + slot * kF8TileBytes);
          const uint32_t p_addr = ptx::smem_u32(smem + Lay::kOffP + (x & 1) * kF8TileBytes);
#pragma unroll
          for (int kk = 0; kk < kTile / 32; ++kk)
            mma_ss_f8(tmem + Lay::kColO, ptx::sdesc_sw128(p_addr + kk * 32, 16, 1024),
                           ptx::sdesc_sw128(vt_addr + kk * 32, 16, 1024), kIdesc, (j > 0 || kk > 0) ? 1u : 0u);
          ptx::mma_commit(o_ready + (x & 1));
          ptx::mma_commit(slot_empty + slot);
          ++pos;
        }
        it += n;
        ++kq;
      }
      ptx::mma_commit(drain);
      ptx::CtaCtl no_abort{0, 0};
      ptx::mbar_wait(drain, 0, &no_abort, nullptr, kSiteFwdDrain, budget);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue (warps 0-3)
    const int r = warp * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float sl = p.s_log2;
    constexpr float kLn2 = 0.6931471805599453f;
    uint8_t* p_row0 = smem + Lay::kOffP + r * 128;  // this row in P buffer 0 (buffer 1: + 16 KB)
    const int sw = r & 7;
    uint32_t it = 0, kq = 0;
    for (int idx = blockIdx.x; idx < n_items; idx += gridDim.x) {
      const Fp8Item I = fp8_item(p, idx);
      const int n = I.n_kv;
      const bool row_ok = kTile * I.t + r < I.L;
      __nv_bfloat16* orow = p.o + (static_cast<int64_t>(I.q_row) + r) * p.heads * kF8D + static_cast<int64_t>(I.h) * kF8D;
      const int64_t lse_i = static_cast<int64_t>(I.h) * p.total + I.q_row + r;
      if (n == 0) {  // no visible key: O = 0, LSE = -inf
        if (row_ok) {
          for (int c = 0; c < kF8D; c += 8) ptx::st_v4(orow + c, 0, 0, 0, 0);
          p.lse[lse_i] = -INFINITY;
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
        // peeled tail: only the diagonal tile (causal) or the end of the keys is masked
        const bool tail = (CAUSAL && j == I.t) || kTile * (j + 1) > I.L;
        if (tail) {
          const int lim = CAUSAL ? min(r + 1 + kTile * (I.t - j), I.L - kTile * j) : I.L - kTile * j;
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
          // rescale O only when the row max grows by more than 2^8 (P stays below 2^8 < 448)
          const bool need = mnew > m + 8.0f;
          if (__any_sync(0xffffffffu, need)) {
            const float mm = need ? mnew : m;
            const float f = ptx::ex2(m - mm);
            const uint32_t xp = x - 1;
            if (!(ok = ptx::mbar_wait(o_ready + (xp & 1), (xp >> 1) & 1, ctl, status, kSiteFwdSoftO, budget))) break;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < kF8D / 32; ++c) {
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
        // P = 2^(s sl - m) as e4m3, 16 keys per 16-byte chunk of the swizzled row
        const float mu = (m == -INFINITY) ? 0.f : m;
        uint8_t* prow = p_row0 + (x & 1) * kF8TileBytes;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t w[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = 16 * ch + 4 * q4 + e;
              pv[e] = ptx::ex2(fmaf(__uint_as_float(sv[col >> 5][col & 31]), sl, -mu));
              l += pv[e];
            }
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(pv[0], pv[1]), __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(pv[2], pv[3]), __NV_SATFINITE, __NV_E4M3);
            w[q4] = lo | (hi << 16);
          }
          ptx::st_shared_v4(prow + ((ch ^ sw) << 4), w[0], w[1], w[2], w[3]);
        }
        ptx::fence_proxy_async_smem();  // the tensor core reads P through the async proxy
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full + (x & 1));
      }
      if (!ok) break;
      // epilogue: O * v_descale / l and LSE for the rows of the sequence
      const uint32_t xl = it + n - 1;
      if (!ptx::mbar_wait(o_ready + (xl & 1), (xl >> 1) & 1, ctl, status, kSiteFwdSoftO, budget)) break;
      ptx::tc_fence_after();
      const float f = l > 0.f ? p.v_descale / l : 0.f;  // a row that sees no key: O = 0
#pragma unroll 1
      for (int c = 0; c < kF8D / 32; ++c) {
        uint32_t ov[32];
        ptx::tmem_ld32(tmem + lane_base + Lay::kColO + 32 * c, ov);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(ov);
        if (row_ok) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wv[e] = ptx::pack_bf16(__uint_as_float(ov[8 * q4 + 2 * e]) * f, __uint_as_float(ov[8 * q4 + 2 * e + 1]) * f);
            ptx::st_v4(orow + 32 * c + 8 * q4, wv[0], wv[1], wv[2], wv[3]);
          }
        }
      }
      if (row_ok) p.lse[lse_i] = (m + log2f(l)) * kLn2;
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

// V (e4m3 [total, H, 128]) -> one [128 head-dim rows x 128 keys] block per key
// tile and head: block (g * H + h) holds key tile g (tile_base numbering) of
// head h, keys past the end of the sequence zero. One CTA per (tile, head).
__global__ void __launch_bounds__(256) vt_transpose_kernel(const uint8_t* __restrict__ v, const int32_t* offsets,
                                                           const int32_t* tile_base, const int32_t* status, int batch,
                                                           int heads, uint8_t* __restrict__ vt) {
  __shared__ __align__(16) uint8_t tile[kTile][kF8D + 16];  // [key][d], padded rows
  const int gt = blockIdx.x, h = blockIdx.y;
  if (status[0] != JFA_OK || gt >= tile_base[batch]) return;
  int lo = 0, hi = batch;  // the sequence of tile gt: largest b with tile_base[b] <= gt
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_base[mid] <= gt) lo = mid; else hi = mid;
  }
  int b = lo;
  while (b + 1 < batch && tile_base[b + 1] <= gt) ++b;
  const int j = gt - tile_base[b];
  const int s0 = offsets[b];
  const int rows = min(kTile, offsets[b + 1] - s0 - kTile * j);  // valid keys of the tile
  for (int k = threadIdx.x; k < kTile * (kF8D / 16); k += blockDim.x) {
    const int key = k / (kF8D / 16), ch = k % (kF8D / 16);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (key < rows)
      val = ptx::ld_nc_v4(v + ((static_cast<int64_t>(s0) + kTile * j + key) * heads + h) * kF8D + 16 * ch);
    *reinterpret_cast<uint4*>(&tile[key][16 * ch]) = val;
  }
  __syncthreads();
  uint8_t* out = vt + (static_cast<int64_t>(gt) * heads + h) * kF8D * kTile;
  for (int k = threadIdx.x; k < kF8D * (kTile / 16); k += blockDim.x) {
    const int d = k / (kTile / 16), kc = k % (kTile / 16);  // head-dim row, 16-key chunk
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int key = 16 * kc + 4 * q;
      w[q] = static_cast<uint32_t>(tile[key][d]) | (static_cast<uint32_t>(tile[key + 1][d]) << 8) |
             (static_cast<uint32_t>(tile[key + 2][d]) << 16) | (static_cast<uint32_t>(tile[key + 3][d]) << 24);
    }
    *reinterpret_cast<uint4*>(out + static_cast<int64_t>(d) * kTile + 16 * kc) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <bool CAUSAL>
cudaError_t launch_fp8_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt, const Fp8Params& p,
                         int grid, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(fwd_fp8_kernel<CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize, Fp8Layout::kAlloc);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  fwd_fp8_kernel<CAUSAL><<<grid, 192, Fp8Layout::kAlloc, stream>>>(tq, tk, tvt, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_vt_transpose(const void* v, const int32_t* offsets, const int32_t* tile_base, const int32_t* status,
                                int batch, int heads, int pad_tiles, void* vt, cudaStream_t stream) {
  dim3 grid(pad_tiles, heads);
  vt_transpose_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(v), offsets, tile_base, status, batch,
                                                heads, static_cast<uint8_t*>(vt));
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const int4* items, const int4* item_seq, int32_t* status, void* o, float* lse, int heads,
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
  return causal ? launch_fp8_t<true>(tq, tk, tvt, p, grid, stream) : launch_fp8_t<false>(tq, tk, tvt, p, grid, stream);
}

}  // namespace jfa
