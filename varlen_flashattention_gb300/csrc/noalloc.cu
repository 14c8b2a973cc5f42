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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "jfa_internal.h"

namespace jfa {
namespace {

constexpr size_t kMaxPartialRows = 32768;  // num_splits * batch * q_heads
constexpr size_t kDecodeScratchBytes = kStatusBytes + kMaxPartialRows * 128 * 4 + kMaxPartialRows * 4;

static __device__ __align__(256) unsigned char g_decode_scratch[kDecodeScratchBytes];

// cuCtxGetCurrent, taken from the driver through the runtime (the library
// does not link libcuda directly).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  return fn;
}

// Scratch addresses already looked up, keyed by CUDA context: the array is
// allocated once per context that loads the library's module, so a context
// recreated after cudaDeviceReset, or a second (non-primary) context on the
// same device, gets its own entry.
constexpr int kMaxContexts = 64;
std::mutex g_mu;
CUcontext g_ctx[kMaxContexts] = {};
void* g_addr[kMaxContexts] = {};
int g_used = 0;

// Device address of g_decode_scratch in the current context (host code cannot
// use the array's name as a device address).
jfa_status scratch_address(void** out) {
  CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (get == nullptr || get(&ctx) != CUDA_SUCCESS) return JFA_ERR_CUDA;
  if (ctx == nullptr) {
    // no context is current yet: the runtime call makes the current device's
    // primary context current
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return JFA_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return JFA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < g_used; ++i)
    if (g_ctx[i] == ctx) {
      *out = g_addr[i];
      return JFA_OK;
    }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return JFA_ERR_CUDA;
  if (g_used < kMaxContexts) {
    g_ctx[g_used] = ctx;
    g_addr[g_used] = p;
    ++g_used;
  }
  *out = p;
  return JFA_OK;
}

}  // namespace
}  // namespace jfa

extern "C" jfa_status jfa_decode_splitkv_noalloc(const jfa_decode_args* args, cudaStream_t stream) {
  // the ordinary argument checks first, so that a bad request reads as such
  // and not as one that is too large
  const jfa_status chk = jfa::check_decode_args(args);
  if (chk != JFA_OK) return chk;
  if (jfa_decode_workspace_size(args) > jfa::kDecodeScratchBytes) return JFA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const jfa_status st = jfa::scratch_address(&scratch);
  if (st != JFA_OK) return st;
  // the decode clears the status block at the start of the call; every
  // partial row it reads is written by the same call first
  return jfa_decode_splitkv(args, scratch, jfa::kDecodeScratchBytes, stream);
}

extern "C" jfa_status jfa_decode_noalloc_status(cudaStream_t stream, int32_t* detail) {
  void* scratch = nullptr;
  const jfa_status st = jfa::scratch_address(&scratch);
  if (st != JFA_OK) return st;
  return jfa_read_device_status(scratch, stream, detail);
}
