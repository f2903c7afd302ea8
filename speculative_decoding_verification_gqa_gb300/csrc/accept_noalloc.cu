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
#include <mutex>

#include "internal.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = SV_ACCEPT_NOALLOC_MAX_WORKSPACE;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_accept_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_accept_scratch, per device

// Device address of the scratch array on the current device. In host code the array's
// name is only a host-side stand-in, so the address is looked up once per device (with
// that device current) and cached.
sv_status scratch_on_current_device(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
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
