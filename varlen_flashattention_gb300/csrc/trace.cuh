// Build-time options of the persistent attention kernels: a per-role event
// trace (JFA_TRACE) and device-side bounds checks of every tile load
// (JFA_DEBUG). The default build compiles both to nothing.
//
// Trace. Warp specialisation splits a CTA into roles (TMA producer, MMA
// issuer, softmax warps, epilogue warps) that hand tiles to one another
// through mbarriers, and a stall in one role shows only as idle time in the
// others ("Cutting-edge isn't plug-and-play: customizing FA4 on B300", bug
// hunting: a producer/consumer pipeline that deadlocked). In a JFA_TRACE
// build every role of the forward-stream and backward kernels records one
// 32-byte record per pipeline event into a buffer the host registers with
// jfa_trace_enable: the SM cycle counter (clock64, comparable between the
// warps of one CTA), the global nanosecond timer, the event (kernel << 16 |
// code), an argument (step or item counter) and the SM id. The buffer address
// and the records per warp reach the kernels through the call's status block,
// written by the status-clear kernel that starts every call. Warp w of CTA b
// writes records [(b * 16 + w) * cap, ... + cap) in order; records past cap
// are dropped. One lane of the warp records.
//
// Checks. In a JFA_DEBUG build the producers check, before each TMA load,
// that the tile's first row lies inside its sequence and its columns inside
// the head's row; a failed check records JFA_ERR_BAD_INPUT with the check's
// site in the status block, raises the CTA's abort flag (every role leaves
// its loop through its bounded waits) and issues no load.
#pragma once

#include <cstdint>

#include "jfa_internal.h"
#include "ptx.cuh"

namespace jfa {
namespace trace {

constexpr int kWarpSlots = 16;      // warp slots per CTA (the kernels have at most 14 warps)
constexpr int kStatusAddr = 16;     // status words 16-17: buffer address (0: recording off)
constexpr int kStatusCap = 18;      // status word 18: records per warp slot
constexpr int kStatusCtas = 19;     // status word 19: CTA slots of the buffer
constexpr int kRecordBytes = 32;

// Events: kernel << 16 | code. Arguments: x = step counter of the CTA (one
// step = one key tile of a forward item, one query tile of a backward item),
// item = item counter of the CTA.
enum Kernel : uint32_t { kFwdStream = 1, kBwd = 2 };
enum FwdEvent : uint32_t {
  kFwdQLoad = 1,       // producer: Q tile of an item issued (item)
  kFwdKVLoad = 2,      // producer: K and V tiles of a step issued (x)
  kFwdSIssue = 3,      // MMA: S = Q K^T issued (x)
  kFwdPVIssue = 4,     // MMA: O += P V issued (x)
  kFwdSoftBegin = 5,   // softmax: S of the step complete (x)
  kFwdSoftEnd = 6,     // softmax: P of the step stored (x)
  kFwdEpiBegin = 7,    // epilogue: O of an item complete (item)
  kFwdEpiEnd = 8,      // epilogue: O and LSE of the item written (item)
  kFwdSoftLoaded = 9,  // softmax: the group's half of S in registers (x)
  kFwdSoftPub = 10,    // softmax: the half's maximum published (x)
  kFwdSoftExp = 11,    // softmax: exponentials taken (the first time) (x)
  kFwdSoftMax = 12,    // softmax: the other half's maximum read (x)
};
enum BwdEvent : uint32_t {
  kBwdKVLoad = 1,      // producer: K and V of an item issued (item)
  kBwdQLoad = 2,       // producer: Q, dO and the LSE / delta rows of a step issued (load counter)
  kBwdItem = 3,        // MMA: K of the item has arrived (item)
  kBwdSIssue = 4,      // MMA: S^T = K Q^T issued (x)
  kBwdDPIssue = 5,     // MMA: dP^T = V dO^T issued (x)
  kBwdDVIssue = 6,     // MMA: dV += P^T dO issued (x)
  kBwdDQDKIssue = 7,   // MMA: dQ = dS K and dK += dS^T Q issued (x)
  kBwdPBegin = 8,      // softmax: S^T complete (x)
  kBwdPEnd = 9,        // softmax: P^T stored (x)
  kBwdDSBegin = 10,    // softmax: dP^T complete and the dS buffer free (x)
  kBwdDSEnd = 11,      // softmax: dS stored (x)
  kBwdDQBegin = 12,    // epilogue: dQ of the step complete (x)
  kBwdDQEnd = 13,      // epilogue: dQ handed to the reduce-adds (x)
  kBwdAccBegin = 14,   // epilogue: dK and dV of the item complete (item)
  kBwdAccEnd = 15,     // epilogue: dK and dV stored (item)
};

#ifdef JFA_TRACE
struct Writer {
  uint8_t* base = nullptr;
  uint32_t cap = 0, n = 0;
  // After the kernel's wait for the previous grid (the status block is written by then).
  __device__ __forceinline__ void open(const int32_t* status, int warp) {
    const uint64_t a = *reinterpret_cast<const volatile unsigned long long*>(status + kStatusAddr);
    cap = static_cast<uint32_t>(status[kStatusCap]);
    if (a != 0 && cap > 0 && warp < kWarpSlots && static_cast<int32_t>(blockIdx.x) < status[kStatusCtas])
      base = reinterpret_cast<uint8_t*>(a) + (static_cast<uint64_t>(blockIdx.x) * kWarpSlots + warp) * cap * kRecordBytes;
  }
  // Called by one lane.
  __device__ __forceinline__ void rec(uint32_t kernel, uint32_t code, uint32_t arg) {
    if (base != nullptr && n < cap) {
      uint32_t sm;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
      const uint64_t clk = clock64();
      const uint64_t gt = ptx::globaltimer();
      uint4* r = reinterpret_cast<uint4*>(base + static_cast<uint64_t>(n) * kRecordBytes);
      r[0] = make_uint4(static_cast<uint32_t>(clk), static_cast<uint32_t>(clk >> 32), static_cast<uint32_t>(gt),
                        static_cast<uint32_t>(gt >> 32));
      r[1] = make_uint4(kernel << 16 | code, arg, sm, 0u);
    }
    ++n;
  }
};
#else
struct Writer {
  __device__ __forceinline__ void open(const int32_t*, int) {}
  __device__ __forceinline__ void rec(uint32_t, uint32_t, uint32_t) {}
};
#endif

#ifdef JFA_DEBUG
// Debug-build check of a tile's position: true when it holds. On failure:
// JFA_ERR_BAD_INPUT, `site` as the detail, and the CTA's abort flag raised.
__device__ __forceinline__ bool tile_check(bool cond, ptx::CtaCtl* ctl, int32_t* status, int site) {
  if (!cond) {
    ctl->abort = 1;
    if (atomicCAS(status, JFA_OK, JFA_ERR_BAD_INPUT) == JFA_OK) atomicExch(status + 1, site);
  }
  return cond;
}
#define JFA_TILE_OK(cond, ctl, status, site) ::jfa::trace::tile_check((cond), (ctl), (status), (site))
#else
#define JFA_TILE_OK(cond, ctl, status, site) true
#endif

}  // namespace trace
}  // namespace jfa
