// Self-test of the failure detection every pipeline kernel relies on.
//
// "Cutting-edge isn't plug-and-play: customizing FA4 on B300" (TwelveLabs),
// bug hunting section: a producer/consumer pipeline that reused a single
// buffer deadlocked, and only on long sequences. Here every mbarrier wait is
// bounded in time: when a wait runs out it records JFA_ERR_TIMEOUT and a site
// code in the workspace status word and raises the CTA's abort flag, which
// the other roles poll so that they leave their loops too; the kernel returns
// and the CUDA context stays usable.
//
// This kernel runs that path on purpose with two roles of a two-stage chain:
// role 0 waits for an input that nothing ever provides (its budget runs out),
// role 1 waits for role 0's output with an eight times longer budget and must
// leave through the abort flag, well before its own budget would.
#include <cuda_runtime.h>

#include <cstdint>

#include "jfa_internal.h"
#include "ptx.cuh"

namespace jfa {

namespace {

__global__ void __launch_bounds__(64) selftest_wait_kernel(int32_t* status, uint64_t budget_ns) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ ptx::CtaCtl ctl;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars[0], 1);
    ptx::mbar_init(&bars[1], 1);
    ctl.abort = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane != 0) return;
  if (warp == 0) {
    // the first stage: its input barrier is never arrived on
    if (ptx::mbar_wait(&bars[0], 0, &ctl, status, kSiteSelftestInput, budget_ns)) ptx::mbar_arrive(&bars[1]);
  } else {
    // the second stage waits for the first; it must see the abort flag
    const uint64_t t0 = ptx::globaltimer();
    const bool ok = ptx::mbar_wait(&bars[1], 0, &ctl, status, kSiteSelftestChain, 8 * budget_ns);
    const uint64_t waited = ptx::globaltimer() - t0;
    status[4] = (!ok && waited < 8 * budget_ns) ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_selftest_wait(int32_t* status, uint64_t budget_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(status, budget_ns);
  return cudaGetLastError();
}

}  // namespace jfa
