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
// the order is deterministic and bit-exact. It also checks the offsets. The
// number of tiles a sequence has in a cost bucket has a closed form, and the
// buckets are dealt to the warps: each warp counts, then places, the tiles of
// its buckets with warp scans over the sequences, and one block scan over the
// bucket totals gives every bucket its start. The work grows with
// buckets x sequences and no step waits on the whole block per bucket.
#include <cuda_runtime.h>

#include <algorithm>

#include "jfa_internal.h"

namespace jfa {

constexpr int kQThreads = 1024;
// Per-sequence values (lengths, first rows, tile bases) kept in shared memory
// for the bucket and record passes, for the first kQueueLenCache sequences
// (longer batches read the rest from global memory).
constexpr int kQueueLenCache = 4 * 1024;

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
// tiles (backward). Lq / Lk are the sequence's query and key lengths (equal
// in the self modes; the broadcast modes pass the key length for both).
__device__ __forceinline__ int item_tiles(const QueueParams& p, int Lq, int Lk) {
  switch (p.mode) {
    case kQueueBcastFwd: return ceil_tiles(p.q_len);
    case kQueueVarFwd: return ceil_tiles(Lq);
    default: return ceil_tiles(Lk);
  }
}

// Varlen, bottom-right causal: key tiles seen by query tile t (a prefix of
// the key tiles: the tile's last row sees keys up to row + L_k - L_q).
__device__ __forceinline__ int var_fwd_tiles(int Lq, int Lk, int t) {
  const int seen = min(kTile * (t + 1), Lq) + Lk - Lq;  // keys visible to the tile's last row
  return seen <= 0 ? 0 : min(ceil_tiles(seen), ceil_tiles(Lk));
}

// Varlen, bottom-right causal: query tiles that see key tile u (a suffix: the
// first query that sees key 128 u is 128 u - (L_k - L_q)).
__device__ __forceinline__ int var_bwd_tiles(int Lq, int Lk, int u) {
  const int i_min = max(0, kTile * u - (Lk - Lq));
  return i_min >= Lq ? 0 : ceil_tiles(Lq) - i_min / kTile;
}

// Partner tiles an item visits: its cost in the longest-first order.
__device__ __forceinline__ int item_cost(const QueueParams& p, int Lq, int Lk, int t) {
  const int nk = ceil_tiles(Lk);
  switch (p.mode) {
    case kQueueSelfFwd: return p.causal ? t + 1 : nk;
    case kQueueSelfBwd: return p.causal ? nk - t : nk;
    case kQueueBcastFwd: return nk;
    case kQueueVarFwd: return p.causal ? var_fwd_tiles(Lq, Lk, t) : nk;
    case kQueueVarBwd: return p.group * (p.causal ? var_bwd_tiles(Lq, Lk, t) : ceil_tiles(Lq));
    default: return ceil_tiles(p.q_len);  // kQueueBcastBwd
  }
}

// First index in [0, n) at which a monotone (false ... true) predicate holds, or n.
template <class F>
__device__ __forceinline__ int first_true(int n, F pred) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pred(mid)) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// Tiles of a sequence with cost k: count, and the first of them (they are
// consecutive: causal self-attention has exactly one tile per cost up to the
// number of tiles; varlen causal costs are monotone in the tile, found by
// binary search; otherwise all tiles share one cost).
__device__ __forceinline__ void tiles_with_cost(const QueueParams& p, int Lq, int Lk, int k, int& count, int& t_first) {
  const int nt = item_tiles(p, Lq, Lk);
  count = 0;
  t_first = 0;
  if (p.causal && (p.mode == kQueueSelfFwd || p.mode == kQueueSelfBwd)) {
    if (k >= 1 && k <= nt) {
      count = 1;
      t_first = (p.mode == kQueueSelfFwd) ? k - 1 : nt - k;
    }
  } else if (p.causal && p.mode == kQueueVarFwd) {  // cost non-decreasing in t
    const int a = first_true(nt, [&](int t) { return item_cost(p, Lq, Lk, t) >= k; });
    const int b = first_true(nt, [&](int t) { return item_cost(p, Lq, Lk, t) >= k + 1; });
    count = b - a;
    t_first = a;
  } else if (p.causal && p.mode == kQueueVarBwd) {  // cost non-increasing in t
    const int a = first_true(nt, [&](int t) { return item_cost(p, Lq, Lk, t) <= k; });
    const int b = first_true(nt, [&](int t) { return item_cost(p, Lq, Lk, t) <= k - 1; });
    count = b - a;
    t_first = a;
  } else if (nt > 0 && item_cost(p, Lq, Lk, 0) == k) {
    count = nt;
  }
}

// Query and key lengths of sequence b (cached in shared memory for the first
// kQueueLenCache sequences).
__device__ __forceinline__ int2 seq_lens(const QueueParams& p, const int* s_len, const int* s_lenk, int b) {
  const int L = b < kQueueLenCache ? s_len[b] : p.offsets[b + 1] - p.offsets[b];
  if (!queue_var(p.mode)) return make_int2(L, L);
  const int Lk = b < kQueueLenCache ? s_lenk[b] : p.k_offsets[b + 1] - p.k_offsets[b];
  return make_int2(L, Lk);
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// kmax: the largest cost. Dynamic shared memory: kmax + 1 bucket starts, then,
// for the first C = min(batch, kQueueLenCache) sequences, the (query) lengths,
// the first queue positions, the first rows and the tile bases, and (varlen)
// the key lengths and first key rows: the record passes then read no global
// memory per sequence (a dependent global load per sequence and warp had
// dominated the kernel).
// The one-pass counting sort (fast path) applies when every tile of a sequence
// has the same cost (not causal), the batch has one sequence per thread and
// the costs fit 32 buckets; it needs a [32 buckets][32 warps] table.
__host__ __device__ inline bool queue_fast_path(const QueueParams& p, int kmax) {
  return !p.causal && p.batch <= 1024 && kmax < 32;
}
constexpr int kQueueFastTable = 32 * 32;

__global__ void __launch_bounds__(kQThreads) build_queue_kernel(const QueueParams p, int kmax) {
  wait_prior_grid();  // the status block is cleared by the kernel before this one
  allow_next_grid();
  extern __shared__ int s_start[];  // [kmax + 1]: tiles (per head) of higher cost than bucket k
  const int n_cached = min(p.batch, kQueueLenCache);
  const bool fast = queue_fast_path(p, kmax);
  // fast path: [bucket][warp] tiles, then their exclusive prefix over warps
  int (*s_wtot)[32] = reinterpret_cast<int (*)[32]>(s_start + kmax + 1);
  int* s_len = s_start + kmax + 1 + (fast ? kQueueFastTable : 0);
  int* s_first = s_len + n_cached;  // first tile position of sequence b (one-cost modes)
  int* s_off = s_first + n_cached;  // first (query) row of sequence b
  int* s_tb = s_off + n_cached;     // tile base of sequence b
  int* s_lenk = s_tb + n_cached;    // varlen: key lengths
  int* s_koff = s_lenk + n_cached;  // varlen: first key row
  const bool var = queue_var(p.mode);
  __shared__ int warp_buf[32];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kQThreads / 32;
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
      if (b < kQueueLenCache) {
        s_len[b] = L;
        s_off[b] = lo;
      }
      if (var) {  // the key offsets obey the same rules
        const int klo = p.k_offsets[b], khi = p.k_offsets[b + 1];
        const int Lk = khi - klo;
        bool kbad = Lk < 0 || Lk > p.max_seqlen_k;
        if (b == 0 && klo != 0) kbad = true;
        if (b == p.batch - 1 && khi != p.total_k) kbad = true;
        if (kbad) s_bad = 1;
        if (b < kQueueLenCache) {
          s_lenk[b] = Lk;
          s_koff[b] = klo;
        }
      }
      nt = bad ? 0 : ceil_tiles(L);
    }
    int tot;
    const int pre = block_exclusive_scan(nt, warp_buf, &tot);
    if (b < p.batch && p.tile_base) p.tile_base[b] = carry + pre;
    if (b < p.batch && b < kQueueLenCache) s_tb[b] = carry + pre;
    carry += tot;
  }
  if (tid == 0 && p.tile_base) p.tile_base[p.batch] = carry;
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      if (atomicCAS(p.status, JFA_OK, JFA_ERR_BAD_INPUT) == JFA_OK) p.status[1] = kSiteQueueOffsets;
      p.status[p.count_index] = 0;
      p.status[p.count_index + 1] = 0;
    }
    return;
  }

  // 2. tiles per cost bucket; warp w takes the buckets kmin + w + 32 i
  // items of cost 0 still own outputs: query rows with no key (O = 0, LSE = -inf),
  // varlen key tiles that no query sees (dK = dV = 0)
  const bool keep_empty = p.mode == kQueueBcastFwd || var;
  const int kmin = keep_empty ? 0 : 1;
  // Fast path (counting sort in one pass, queue_fast_path): each sequence's
  // bucket and tile count are found once, and the per-bucket totals and
  // positions come from shared-memory sums and warp scans, instead of one pass
  // over all sequences per bucket.
  int f_k = -1, f_c = 0;          // fast path: this thread's sequence's bucket and tiles (0: none queued)
  if (fast) {
    s_wtot[warp][lane] = 0;
    if (tid <= kmax) s_start[tid] = 0;
    if (tid < p.batch) {
      const int2 L = seq_lens(p, s_len, s_lenk, tid);
      const int nt = item_tiles(p, L.x, L.y);
      const int k = nt > 0 ? item_cost(p, L.x, L.y, 0) : -1;
      if (nt > 0 && k >= kmin) {
        f_k = k;
        f_c = nt;
      }
    }
    __syncthreads();
    if (f_c > 0) {
      atomicAdd(&s_start[f_k], f_c);
      atomicAdd(&s_wtot[f_k][warp], f_c);
    }
  } else {
    for (int k = kmin + warp; k <= kmax; k += kWarps) {
      int n = 0;
      for (int b = lane; b < p.batch; b += 32) {
        int c, tf;
        const int2 L = seq_lens(p, s_len, s_lenk, b);
        tiles_with_cost(p, L.x, L.y, k, c, tf);
        n += c;
      }
      n = warp_sum(n);
      if (lane == 0) s_start[k] = n;
    }
  }
  __syncthreads();

  // 3. bucket starts in descending cost order
  int total_tiles = 0;
  for (int k0 = kmax; k0 >= kmin; k0 -= kQThreads) {
    const int k = k0 - tid;
    const int v = k >= kmin ? s_start[k] : 0;
    int tot;
    const int pre = block_exclusive_scan(v, warp_buf, &tot);
    if (k >= kmin) s_start[k] = total_tiles + pre;
    total_tiles += tot;
  }
  __syncthreads();
  // tiles with cost >= 1 come first
  const int busy_tiles = kmin == 0 ? s_start[0] : total_tiles;

  // 4. place the items: within a bucket ascending (b, tile, h). When all tiles
  // of a sequence share one cost, the bucket pass only records where each
  // sequence starts, and the records are then written by every warp for its
  // own sequences (below), so that one large bucket is not written by one warp.
  const bool one_cost = !p.causal;  // the broadcast modes are never causal
  // The items fit the queue (checked once here; every write below is in range).
  const bool fits = static_cast<int64_t>(total_tiles) * p.heads <= p.max_items;
  // a sequence's first row, first key row and tile base, from shared memory when cached
  auto row0 = [&](int b) { return b < kQueueLenCache ? s_off[b] : p.offsets[b]; };
  auto krow0 = [&](int b) { return b < kQueueLenCache ? s_koff[b] : p.k_offsets[b]; };
  auto tbase = [&](int b) { return p.tile_base ? (b < kQueueLenCache ? s_tb[b] : p.tile_base[b]) : 0; };
  auto write_items = [&](int b, int first, int c, int tf, int k, int2 L) {
    if (!fits) return;
    const int tb = tbase(b);
    const int4 seq = var ? make_int4(row0(b), L.x, krow0(b), L.y) : make_int4(row0(b), L.x, tb, 0);
    const int w = p.mode == kQueueVarBwd ? tb : k;  // the varlen backward carries the query tile base
    int4* it = p.items + static_cast<int64_t>(first) * p.heads;
    int4* sq = p.item_seq ? p.item_seq + static_cast<int64_t>(first) * p.heads : nullptr;
    for (int r = 0; r < c; ++r)
      for (int h = 0; h < p.heads; ++h) *it++ = make_int4(b, h, tf + r, w);
    if (sq)
      for (int e = 0; e < c * p.heads; ++e) *sq++ = seq;
  };
  if (fast) {
    // the tiles of earlier warps in each bucket (warp k scans bucket k over the
    // warps), then of earlier lanes with the same bucket in this warp
    if (warp <= kmax) {
      const int v = s_wtot[warp][lane];
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      s_wtot[warp][lane] = incl - v;
    }
    int pre = 0;
#pragma unroll 8
    for (int j = 0; j < 32; ++j) {
      const int kj = __shfl_sync(0xffffffffu, f_k, j), cj = __shfl_sync(0xffffffffu, f_c, j);
      if (j < lane && kj == f_k) pre += cj;
    }
    __syncthreads();
    if (f_c > 0) s_first[tid] = s_start[f_k] + s_wtot[f_k][warp] + pre;
  }
  for (int k = kmin + warp; !fast && k <= kmax; k += kWarps) {
    int run = s_start[k];
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
      const int b = b0 + lane;
      int c = 0, tf = 0;
      int2 L = make_int2(0, 0);
      if (b < p.batch) {
        L = seq_lens(p, s_len, s_lenk, b);
        tiles_with_cost(p, L.x, L.y, k, c, tf);
      }
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const int first = run + incl - c;
      run += __shfl_sync(0xffffffffu, incl, 31);
      if (c > 0) {
        if (one_cost && b < kQueueLenCache)
          s_first[b] = first;  // written below by the thread that owns b
        else
          write_items(b, first, c, tf, k, L);
      }
    }
  }
  if (one_cost) {
    // Each thread works out its own sequence's records once (first position,
    // count, cost word, bounds); then every warp writes the records of its 32
    // sequences one sequence at a time, the values broadcast from the owning
    // lane and one record per lane, so each store instruction covers up to 32
    // consecutive records and no lane repeats the per-sequence arithmetic (a
    // warp per sequence with every lane recomputing it made this loop
    // instruction-bound, ~3/4 of the kernel).
    __syncthreads();
    const int n_seq = min(p.batch, kQueueLenCache);
    const int t_lane = lane / p.heads, h_lane = lane - t_lane * p.heads;  // record `lane` of a sequence
    for (int b0 = 0; b0 < n_seq; b0 += kQThreads) {
      const int b = b0 + tid;
      int first = 0, n = 0, w = 0;
      int4 seq = make_int4(0, 0, 0, 0);
      if (b < n_seq) {
        const int2 L = seq_lens(p, s_len, s_lenk, b);
        const int nt = item_tiles(p, L.x, L.y);
        const int k = nt > 0 ? item_cost(p, L.x, L.y, 0) : 0;
        if (fits && nt > 0 && k >= kmin) {
          const int tb = tbase(b);
          seq = var ? make_int4(row0(b), L.x, krow0(b), L.y) : make_int4(row0(b), L.x, tb, 0);
          w = p.mode == kQueueVarBwd ? tb : k;
          first = s_first[b];
          n = nt * p.heads;  // records tile-major, heads inner: record e = (tile e / H, head e % H)
        }
      }
      for (int j = 0; j < 32; ++j) {
        const int nj = __shfl_sync(0xffffffffu, n, j);
        if (nj == 0) continue;
        const int bj = b0 + 32 * warp + j;
        const int64_t fj = static_cast<int64_t>(__shfl_sync(0xffffffffu, first, j)) * p.heads;
        const int wj = __shfl_sync(0xffffffffu, w, j);
        const int4 sj = make_int4(__shfl_sync(0xffffffffu, seq.x, j), __shfl_sync(0xffffffffu, seq.y, j),
                                  __shfl_sync(0xffffffffu, seq.z, j), __shfl_sync(0xffffffffu, seq.w, j));
        for (int e = lane; e < nj; e += 32) {
          int t = t_lane, h = h_lane;
          if (e != lane) {
            t = e / p.heads;
            h = e - t * p.heads;
          }
          p.items[fj + e] = make_int4(bj, h, t, wj);
          if (p.item_seq) p.item_seq[fj + e] = sj;
        }
      }
    }
  }
  if (tid == 0) {
    int64_t n_items = static_cast<int64_t>(total_tiles) * p.heads;
    int64_t n_busy = static_cast<int64_t>(busy_tiles) * p.heads;
    if (!fits) {
      if (atomicCAS(p.status, JFA_OK, JFA_ERR_BAD_INPUT) == JFA_OK) p.status[1] = kSiteQueueOffsets;
      n_items = 0;
      n_busy = 0;
    }
    p.status[p.count_index] = static_cast<int32_t>(n_items);
    p.status[p.count_index + 1] = static_cast<int32_t>(n_busy);
  }
}

// The largest cost bucket the queue handles (its starts live in shared memory).
constexpr int kQueueMaxCost = 32 * 1024;

cudaError_t launch_queue(const QueueParams& p, cudaStream_t stream) {
  auto tiles = [](int64_t L) { return (L + kTile - 1) / kTile; };
  int64_t kmax = tiles(p.max_seqlen);
  if (p.mode == kQueueBcastBwd) kmax = tiles(p.q_len);
  if (p.mode == kQueueVarFwd) kmax = tiles(p.max_seqlen_k);
  if (p.mode == kQueueVarBwd) kmax = static_cast<int64_t>(p.group) * tiles(p.max_seqlen);
  if (kmax > kQueueMaxCost) return cudaErrorInvalidValue;
  const int64_t cached = std::min(p.batch, kQueueLenCache);
  const int64_t table = queue_fast_path(p, static_cast<int>(kmax)) ? kQueueFastTable : 0;
  const size_t smem = static_cast<size_t>(kmax + 1 + table + cached * (queue_var(p.mode) ? 6 : 4)) * sizeof(int);
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(build_queue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>((kQueueMaxCost + 1 + 6 * kQueueLenCache) * sizeof(int)));
  });
  if (e != cudaSuccess) return e;
  return launch_after(build_queue_kernel, dim3(1), dim3(kQThreads), smem, stream, p, static_cast<int>(kmax));
}

// A call's status block cleared by one small block; the call's next kernel may
// be scheduled at once (it waits for this one before reading the block).
#ifdef JFA_TRACE
namespace {
std::atomic<uint64_t> g_trace_addr{0};
std::atomic<int32_t> g_trace_cap{0};
std::atomic<int32_t> g_trace_ctas{0};
}  // namespace

void set_trace_buffer(void* buffer, int32_t records_per_warp, int32_t ctas) {
  g_trace_cap.store(buffer ? records_per_warp : 0);
  g_trace_ctas.store(buffer ? ctas : 0);
  g_trace_addr.store(reinterpret_cast<uint64_t>(buffer));
}

// Also writes the registered trace buffer into status words 16-19, where the
// persistent kernels of the call read it.
__global__ void status_clear_kernel(int32_t* status, uint64_t trace_addr, int32_t trace_cap, int32_t trace_ctas) {
  allow_next_grid();
  int32_t w = 0;
  if (threadIdx.x == 16) w = static_cast<int32_t>(static_cast<uint32_t>(trace_addr));
  if (threadIdx.x == 17) w = static_cast<int32_t>(static_cast<uint32_t>(trace_addr >> 32));
  if (threadIdx.x == 18) w = trace_cap;
  if (threadIdx.x == 19) w = trace_ctas;
  status[threadIdx.x] = w;
}

cudaError_t launch_status_clear(int32_t* status, cudaStream_t stream) {
  status_clear_kernel<<<1, kStatusBytes / 4, 0, stream>>>(status, g_trace_addr.load(), g_trace_cap.load(),
                                                        g_trace_ctas.load());
  return cudaGetLastError();
}
#else
__global__ void status_clear_kernel(int32_t* status) {
  allow_next_grid();
  status[threadIdx.x] = 0;
}

cudaError_t launch_status_clear(int32_t* status, cudaStream_t stream) {
  status_clear_kernel<<<1, kStatusBytes / 4, 0, stream>>>(status);
  return cudaGetLastError();
}
#endif

}  // namespace jfa
