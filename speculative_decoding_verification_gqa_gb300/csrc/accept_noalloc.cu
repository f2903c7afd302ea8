// accept_noalloc.cu -- spec_accept for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: inference engines that
// reserve all of their device memory once at start-up and then give each operator only
// its inputs and outputs (plugin-style interfaces without a scratch argument), so any
// per-call cudaMalloc would break their memory plan. For them, spec_accept_noalloc keeps
// the acceptance step's scratch (one (value, index) key per window row, a completion
// ticket, the flag word) in a fixed array compiled into the library.
//
// Cost and limits: every GPU that loads the library holds kNoallocScratchBytes of device
// memory until the process exits; shapes that need more scratch are rejected. All calls
// share the one array per device, so calls that can overlap on the GPU race.
#include <cuda.h>

#include <mutex>

#include "internal.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = SV_ACCEPT_NOALLOC_MAX_WORKSPACE;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_accept_scratch[kNoallocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Driver entry points, fetched through the runtime (the library links no libcuda).
template <class Fn>
Fn driver_fn(const char* name) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return (Fn)f;
}

// Unique id of the calling thread's current context (0 if there is none yet).
bool current_ctx_id(unsigned long long* id) {
  static CtxGetCurrentFn get_cur = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_cur || !get_id) return false;
  CUcontext c = nullptr;
  if (get_cur(&c) != CUDA_SUCCESS) return false;
  if (!c) {
    *id = 0;
    return true;
  }
  return get_id(c, id) == CUDA_SUCCESS;
}

struct ScratchEntry {
  unsigned long long ctx;  // context the address belongs to
  void* addr;              // device address of g_accept_scratch in it
};
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxDevices];

// Device address of the scratch array in the current device's current context. In host
// code the array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress and cached per device, together with the id of the context it
// belongs to: after cudaDeviceReset (or any new primary context) the id changes and the
// address is looked up again in the new context, whose copy of the array starts at zero.
sv_status scratch_on_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long ctx = 0;
  if (!current_ctx_id(&ctx)) return SV_ERR_CUDA;
  if (ctx == 0 || g_scratch[dev].ctx != ctx || !g_scratch[dev].addr) {
    void* p = nullptr;  // (makes the device's primary context current if there was none)
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
    if (!current_ctx_id(&ctx) || ctx == 0) return SV_ERR_CUDA;
    g_scratch[dev] = ScratchEntry{ctx, p};
  }
  *addr = g_scratch[dev].addr;
  return SV_OK;
}

}  // namespace

extern "C" SV_API sv_status spec_accept_noalloc(int32_t batch, int32_t max_draft_len,
                                                int32_t vocab, int32_t logits_dtype,
                                                const void* logits,
                                                const int32_t* draft_tokens,
                                                const int32_t* draft_len, int32_t* accept_len,
                                                int32_t* next_token, int32_t* target_tokens,
                                                void* stream) {
  void* scratch = nullptr;
  const sv_status st = scratch_on_current_device(&scratch);
  if (st != SV_OK) return st;
  // Same checks and kernels as spec_accept; a shape whose scratch exceeds the array fails
  // its workspace-size check with SV_ERR_WORKSPACE before anything is launched. The array
  // starts at zero (static storage) and every call leaves it at zero apart from the flag
  // word, which is only ever OR-ed into.
  return spec_accept(batch, max_draft_len, vocab, logits_dtype, logits, draft_tokens,
                     draft_len, accept_len, next_token, target_tokens, scratch,
                     kNoallocScratchBytes, stream);
}
