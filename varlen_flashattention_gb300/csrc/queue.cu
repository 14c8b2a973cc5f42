// Longest-first work queue for the persistent attention kernels.
//
// "Optimizing Jagged Flash Attention with TLX" (aivexanews), fourth and fifth
// paragraphs: both passes are persistent (one CTA per SM looping over tiles)
// and software load balancing of the jagged tiles recovers ~20% of the
// forward. The page does not give the balancing rule; the one used here:
// items are tiles of 128 rows, ordered by descending cost (the number of
// partner tiles the item has to visit), ties by ascending (b, tile, h), and
// dealt round-robin to the persistent CTAs, so every CTA takes one of the most
// expensive remaining items before any cheaper one.
//
// One CTA builds the whole queue with a bucket (counting) sort on the cost, so
// the order is deterministic and bit-exact. It also checks the offsets.
#include <cuda_runtime.h>

#include "jfa_internal.h"

namespace jfa {

constexpr int kQThreads = 1024;

// Exclusive block-wide scan of one int per thread; returns the prefix and
// writes the block total to *total. All kQThreads threads must call it.
__device__ int block_exclusive_scan(int v, int* warp_buf, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_buf[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    warp_buf[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp == 0 ? 0 : warp_buf[warp - 1]) + x - v;
  *total = warp_buf[31];
  __syncthreads();
  return before;
}

__device__ __forceinline__ int ceil_tiles(int L) { return (L + kTile - 1) / kTile; }

// Work items of sequence b (per head): query tiles (forward) or key/value
// tiles (backward).
__device__ __forceinline__ int item_tiles(const QueueParams& p, int L) {
  return p.mode == kQueueBcastFwd ? ceil_tiles(p.q_len) : ceil_tiles(L);
}

// Partner tiles an item visits: its cost in the longest-first order.
__device__ __forceinline__ int item_cost(const QueueParams& p, int L, int t) {
  const int nk = ceil_tiles(L);
  switch (p.mode) {
    case kQueueSelfFwd: return p.causal ? t + 1 : nk;
    case kQueueSelfBwd: return p.causal ? nk - t : nk;
    case kQueueBcastFwd: return nk;
    default: return ceil_tiles(p.q_len);  // kQueueBcastBwd
  }
}

__global__ void __launch_bounds__(kQThreads) build_queue_kernel(const QueueParams p) {
  __shared__ int warp_buf[32];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // 1. validate offsets, prefix sum of 128-row tiles per sequence
  int carry = 0;
  for (int b0 = 0; b0 < p.batch; b0 += kQThreads) {
    const int b = b0 + tid;
    int nt = 0;
    if (b < p.batch) {
      const int lo = p.offsets[b], hi = p.offsets[b + 1];
      const int L = hi - lo;
      bool bad = L < 0 || L > p.max_seqlen;
      if (b == 0 && lo != 0) bad = true;
      if (b == p.batch - 1 && hi != p.total) bad = true;
      if (bad) s_bad = 1;
      nt = bad ? 0 : ceil_tiles(L);
    }
    int tot;
    const int pre = block_exclusive_scan(nt, warp_buf, &tot);
    if (b < p.batch && p.tile_base) p.tile_base[b] = carry + pre;
    carry += tot;
  }
  if (tid == 0 && p.tile_base) p.tile_base[p.batch] = carry;
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      if (atomicCAS(p.status, JFA_OK, JFA_ERR_BAD_INPUT) == JFA_OK) p.status[1] = kSiteQueueOffsets;
      p.status[p.count_index] = 0;
    }
    return;
  }

  // 2. bucket sort by descending cost; within a cost, ascending (b, tile, h)
  const int kmax = (p.mode == kQueueBcastBwd) ? ceil_tiles(p.q_len) : ceil_tiles(p.max_seqlen);
  const bool keep_empty = p.mode == kQueueBcastFwd;  // empty K/V still owns output rows
  const int kmin = keep_empty ? 0 : 1;
  int base = 0;
  for (int k = kmax; k >= kmin; --k) {
    int bucket = 0;
    for (int b0 = 0; b0 < p.batch; b0 += kQThreads) {
      const int b = b0 + tid;
      // Tiles of sequence b with cost k, in ascending order: t_first and count,
      // in closed form (causal: exactly one tile; otherwise all tiles share one
      // cost).
      int count = 0, L = 0, nt = 0, t_first = 0;
      if (b < p.batch) {
        L = p.offsets[b + 1] - p.offsets[b];
        nt = item_tiles(p, L);
        if (p.causal && (p.mode == kQueueSelfFwd || p.mode == kQueueSelfBwd)) {
          count = (k <= nt) ? 1 : 0;
          t_first = (p.mode == kQueueSelfFwd) ? k - 1 : nt - k;
        } else {
          count = (nt > 0 && item_cost(p, L, 0) == k) ? nt : 0;
        }
      }
      int tot;
      const int pre = block_exclusive_scan(count, warp_buf, &tot);
      int r = 0;
      for (int t = t_first; t < nt && r < count; ++t) {
        const int slot = base + (bucket + pre + r) * p.heads;
        for (int h = 0; h < p.heads; ++h) {
          if (slot + h < p.max_items) p.items[slot + h] = make_int4(b, h, t, k);
        }
        ++r;
      }
      bucket += tot;
    }
    base += bucket * p.heads;
  }
  if (tid == 0) {
    if (base > p.max_items) {
      if (atomicCAS(p.status, JFA_OK, JFA_ERR_BAD_INPUT) == JFA_OK) p.status[1] = kSiteQueueOffsets;
      base = 0;
    }
    p.status[p.count_index] = base;
  }
}

cudaError_t launch_queue(const QueueParams& p, cudaStream_t stream) {
  build_queue_kernel<<<1, kQThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace jfa
