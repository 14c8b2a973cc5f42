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

// Number of tiles (work items per head) of sequence b, and the cost of tile t.
__device__ __forceinline__ int item_tiles(const QueueParams& p, int L) {
  return p.mode == kQueueBcastFwd ? ceil_tiles(p.q_len) : ceil_tiles(L);
}

__global__ void __launch_bounds__(kQThreads) build_queue_kernel(const QueueParams p) {
  __shared__ int warp_buf[32];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = 0;
  __syncthreads();

  const bool self = (p.mode == kQueueSelfFwd || p.mode == kQueueSelfBwd);
  // 1. validate offsets, prefix sum of tiles per sequence
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
      p.status[2] = 0;
    }
    return;
  }

  // 2. bucket sort by descending cost
  int kmax;
  if (p.mode == kQueueBcastBwd)
    kmax = ceil_tiles(p.q_len);
  else
    kmax = ceil_tiles(p.max_seqlen);
  const int kmin = (p.mode == kQueueBcastFwd) ? 0 : 1;  // an empty K/V sequence still owns output rows
  int base = 0;
  for (int k = kmax; k >= kmin; --k) {
    int bucket = 0;
    for (int b0 = 0; b0 < p.batch; b0 += kQThreads) {
      const int b = b0 + tid;
      int count = 0, L = 0, nt = 0;
      if (b < p.batch) {
        L = p.offsets[b + 1] - p.offsets[b];
        nt = item_tiles(p, L);
        if (self && p.causal) {
          count = (nt >= k) ? 1 : 0;  // fwd: tile k-1; bwd: tile nt-k
        } else {
          int cost;
          if (p.mode == kQueueBcastFwd)
            cost = ceil_tiles(L);
          else if (p.mode == kQueueBcastBwd)
            cost = ceil_tiles(p.q_len);
          else
            cost = nt;
          count = (cost == k) ? nt : 0;
        }
      }
      int tot;
      const int pre = block_exclusive_scan(count, warp_buf, &tot);
      for (int r = 0; r < count; ++r) {
        int t;
        if (self && p.causal)
          t = (p.mode == kQueueSelfFwd) ? k - 1 : nt - k;
        else
          t = r;
        const int slot = base + (bucket + pre + r) * p.heads;
        for (int h = 0; h < p.heads; ++h) {
          if (slot + h < p.max_items) p.items[slot + h] = make_int4(b, h, t, k);
        }
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
    p.status[2] = base;
  }
}

cudaError_t launch_queue(const QueueParams& p, cudaStream_t stream) {
  build_queue_kernel<<<1, kQThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace jfa
