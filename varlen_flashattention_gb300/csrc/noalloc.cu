// Paged split-KV decode for callers that cannot allocate device memory.
//
// jfa_decode_splitkv needs a caller-provided workspace for its per-split
// partial results. Some callers cannot provide one at call time: a plugin
// that a host runtime invokes with nothing but its input and output buffers,
// or a latency-critical serving path whose device memory is planned up front
// and where an allocation (and the synchronisation that freeing implies) is
// not allowed. For them this file keeps the scratch in a fixed, file-scope
// device array and runs the ordinary decode on it.
//
// The array is kDecodeScratchBytes (about 16.1 MiB): room for
// num_splits * batch * q_heads <= 32768 partial rows. Every GPU that loads
// the library holds it until the process exits. All calls share it, so calls
// whose work overlaps on the GPU (different streams, or different host
// threads on the same device) race on it; serialise them.
#include <cuda_runtime.h>

#include <mutex>

#include "jfa_internal.h"

namespace jfa {
namespace {

constexpr size_t kMaxPartialRows = 32768;  // num_splits * batch * q_heads
constexpr size_t kDecodeScratchBytes = kStatusBytes + kMaxPartialRows * 128 * 4 + kMaxPartialRows * 4;

static __device__ __align__(256) unsigned char g_decode_scratch[kDecodeScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, looked up once
// per device (host code cannot use the array's name as a device address).
jfa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return JFA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return JFA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return JFA_OK;
}

}  // namespace
}  // namespace jfa

extern "C" jfa_status jfa_decode_splitkv_noalloc(const jfa_decode_args* args, cudaStream_t stream) {
  if (!args) return JFA_ERR_INVALID_ARG;
  if (jfa_decode_workspace_size(args) > jfa::kDecodeScratchBytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const jfa_status st = jfa::scratch_address(&scratch);
  if (st != JFA_OK) return st;
  // the decode clears the status block at the start of the call; every
  // partial row it reads is written by the same call first
  return jfa_decode_splitkv(args, scratch, jfa::kDecodeScratchBytes, stream);
}
