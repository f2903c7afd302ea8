// attn_tc.cu -- verify attention on the fifth-generation tensor cores (tcgen05).
// Not built yet: the selector falls back to the mma.sync kernel.
#include "internal.cuh"

namespace sv {

bool attn_tc_available() { return false; }
int attn_tc_kt() { return 128; }
cudaError_t launch_attn_tc(const AttnParams&, bool, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace sv
